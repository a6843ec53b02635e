// scan_pipe_kernel.cuh -- persistent, warp-specialised form of the fused
// score + chunked prefix scan for bfloat16 K and V (the path of the long,
// HBM-bound workloads): the many-to-many softmax-attention output in one pass
// over K and V.
//
// The method is the one of scan_kernel.cuh ("Attention as an RNN" review,
// "Proposed method": every prefix output o_t is the inclusive prefix of the
// associative (m, u, w) operator; "Self-attention Does Not Need O(n^2)
// Memory" review, sections 2 and 3: running sums kept stable by the running
// maximum).  What differs is how the work is laid out on an SM.
//
// One block per SM stays alive for the whole launch.  It holds GROUPS
// independent groups that share a small pool of shared-memory stages (K, V
// and q of a 128-token chunk each); each group has five warps:
//   * four compute warps; warp w owns tokens [32w, 32w + 32) of the chunk:
//       - scores, lane = token: bfloat16 keys with the mixed-precision FMA,
//         float32 keys with the compensated dot product (the functions the
//         other kernels use, so every kernel sees the same scores);
//       - V of the warp's rows is copied into registers (lane l owns dims
//         [E l, E l + E)), the stage is handed back ("empty" mbarrier), and
//         the warp aggregate (m, u, w) goes to shared memory ("agg");
//       - compute warp 1 combines the four warp aggregates into the chunk
//         aggregate, hands it to the carry warp ("cagg") and publishes it for
//         successors' look-backs;
//       - once the chunk's carry arrives ("carry"), each warp adds the
//         aggregates of the warps before it, rescans from registers and
//         writes O;
//   * one carry warp that never holds V:
//       - claims a stage, takes the group's next chunk ticket (interleaved
//         over heads: ticket = c * heads + head) and issues the 1-D bulk
//         copies (TMA) of K, V and q;
//       - runs the decoupled look-back over predecessor chunks while the
//         compute warps are still scoring; the predecessors' states come
//         into a fold buffer of the group by bulk copies, one round trip to
//         L2 per window;
//       - hands the chunk's exclusive prefix to the compute warps, takes the
//         group's next ticket (claiming a stage and starting its copies), and
//         then publishes this chunk's inclusive prefix.
// Taking a ticket only when the group is about to need it keeps chunks
// flowing close to ticket order, so predecessors have usually published by
// the time a chunk looks back; the load of the next chunk overlaps the
// rescan of the current one.  Keeping V out of the carry warp keeps the
// register peak to the larger of the two roles.
//
// Forward progress: a ticket is taken only with a stage in hand, and its
// copy is issued at once; every group handles its chunks in ticket order, and
// between taking a ticket and publishing the previous chunk's inclusive
// prefix the carry warp waits on nothing.  The smallest unfinished ticket is
// then always one its group is working on, and it waits only on smaller
// (finished) tickets.  Every wait is bounded (%globaltimer); a wait that
// gives up sets a bit of the device status word and the group stops.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>
#include <type_traits>

#include "common.cuh"
#include "ptx.cuh"
#include "scan_kernel.cuh"

namespace aaren {

constexpr int kPipeComputeWarps = 4;
constexpr int kPipeGroupWarps = kPipeComputeWarps + 1;
// rows per unrolled block of the rescan loop (32: fully unrolled)
#ifndef AAREN_PIPE_RESCAN_BLOCK
#define AAREN_PIPE_RESCAN_BLOCK 4
#endif
constexpr int kRescanBlock = AAREN_PIPE_RESCAN_BLOCK;
// predecessor states a look-back fold brings into shared memory at once, at
// most (fewer where the stages leave less room)
#ifndef AAREN_PIPE_FOLD_SLOTS
#define AAREN_PIPE_FOLD_SLOTS 24
#endif
constexpr int kFoldSlotsMax = AAREN_PIPE_FOLD_SLOTS;
constexpr size_t kSmemPerBlock = 227 * 1024;   // opt-in shared memory of a block
static_assert(32 % kRescanBlock == 0, "rescan blocks must tile the warp's 32 rows");

template <int D, int GROUPS_, int STAGES_, typename Tin_ = __nv_bfloat16>
struct PipeTile {
    using Tin = Tin_;
    static constexpr int GROUPS = GROUPS_;
    static constexpr int STAGES = STAGES_;
    static constexpr int C = 32 * kPipeComputeWarps;   // tokens per chunk
    static constexpr int THREADS = 32 * kPipeGroupWarps * GROUPS;
    static constexpr int SS = StateLayout<D>::SS;
    static constexpr size_t half_bytes = size_t(C) * D * sizeof(Tin);   // K (or V) of a chunk
    static constexpr size_t q_bytes = size_t(D) * sizeof(Tin);
    // A stage of the block's pool: K | V | q of one chunk.
    static constexpr size_t st_v = half_bytes;
    static constexpr size_t st_q = 2 * half_bytes;
    static constexpr size_t stage_bytes = st_q + (q_bytes + 15) / 16 * 16;
    // Per group: warp aggregates (two sets, by chunk parity: compute warp 0
    // may still read a chunk's aggregates to publish them while the other
    // warps write the next chunk's), warp carries, rescan coefficients, the
    // group's current chunk (ticket, stage, fill parity), failure word and
    // four mbarriers.
    static constexpr size_t g_wst = 0;
    static constexpr size_t g_cst = g_wst + 2 * size_t(kPipeComputeWarps) * SS * sizeof(float);
    static constexpr size_t g_coef = g_cst + size_t(kPipeComputeWarps) * SS * sizeof(float);
    static constexpr size_t g_meta = g_coef + size_t(kPipeComputeWarps) * 32 * sizeof(float4);
    static constexpr size_t g_bars = g_meta + 16;
    static constexpr size_t group_bytes = g_bars + 6 * sizeof(uint64_t);   // 5 used, 16-byte multiple
    // Block: the stages, the groups, then the pool's free mask, the stages'
    // fill counters and their "full" mbarriers.
    static constexpr size_t group_off = size_t(STAGES) * stage_bytes;
    static constexpr size_t pool_off = group_off + size_t(GROUPS) * group_bytes;
    static constexpr size_t fills_off = pool_off + 16;
    static constexpr size_t full_off = fills_off + (size_t(STAGES) * 4 + 7) / 8 * 8;
    // each group's look-back fold buffer: FOLD predecessor states, as many
    // as the room the stages leave allows, up to kFoldSlotsMax
    static constexpr size_t fold_off = (full_off + size_t(STAGES) * sizeof(uint64_t) + 15) / 16 * 16;
    static constexpr size_t fold_room = kSmemPerBlock > fold_off ? kSmemPerBlock - fold_off : 0;
    static constexpr int FOLD_FIT = int(fold_room / (size_t(GROUPS) * SS * sizeof(float)));
    static constexpr int FOLD = FOLD_FIT < kFoldSlotsMax ? FOLD_FIT : kFoldSlotsMax;
    static constexpr size_t fold_bytes = size_t(FOLD) * SS * sizeof(float);
    static constexpr size_t smem_bytes = fold_off + size_t(GROUPS) * fold_bytes;
    static_assert(FOLD >= 4 && FOLD <= 32, "the look-back fold needs a few slots, and takes at most one window");
    static_assert(half_bytes % 16 == 0 && stage_bytes % 16 == 0 && g_cst % 16 == 0 &&
                      g_coef % 16 == 0 && g_meta % 16 == 0 && group_bytes % 16 == 0 &&
                      group_off % 16 == 0 && full_off % 8 == 0 && fold_bytes % 16 == 0,
                  "shared-memory regions must stay aligned");
    static_assert(STAGES >= 1 && STAGES <= 32, "the pool's free mask is one word");
    static_assert(smem_bytes <= 227 * 1024, "stages do not fit in shared memory");
};

constexpr long long kTicketStop = -1;   // no chunk left for this group

// E bfloat16 values of one row held in registers (lane-owned dims).
template <int E>
struct RawRow {
    unsigned w[E == 4 ? 2 : 1];
};

// E float32 values of one row held in registers (float32 keys and values).
template <int E>
struct RawRowF {
    float v[E];
};

template <typename Tin, int E>
using PipeRow = typename std::conditional<sizeof(Tin) == 4, RawRowF<E>, RawRow<E>>::type;

template <int E>
__device__ __forceinline__ void lds_row(const float *p, RawRowF<E> &r)
{
    if constexpr (E == 4) {
        const float4 v = *reinterpret_cast<const float4 *>(p);
        r.v[0] = v.x; r.v[1] = v.y; r.v[2] = v.z; r.v[3] = v.w;
    } else if constexpr (E == 2) {
        const float2 v = *reinterpret_cast<const float2 *>(p);
        r.v[0] = v.x; r.v[1] = v.y;
    } else {
        r.v[0] = *p;
    }
}

template <int E>
__device__ __forceinline__ void zero_row(RawRowF<E> &r)
{
#pragma unroll
    for (int e = 0; e < E; ++e) r.v[e] = 0.f;
}

template <int E>
__device__ __forceinline__ void zero_row(RawRow<E> &r)
{
#pragma unroll
    for (int k = 0; k < (E == 4 ? 2 : 1); ++k) r.w[k] = 0u;
}

// float32 rows need no unpacking (the zero register is unused)
template <int E>
__device__ __forceinline__ void unpack_row_late(const RawRowF<E> &r, unsigned, float (&f)[E])
{
#pragma unroll
    for (int e = 0; e < E; ++e) f[e] = r.v[e];
}

template <int E>
__device__ __forceinline__ void lds_row(const __nv_bfloat16 *p, RawRow<E> &r)
{
    if constexpr (E == 4) {
        const uint2 v = *reinterpret_cast<const uint2 *>(p);
        r.w[0] = v.x;
        r.w[1] = v.y;
    } else if constexpr (E == 2) {
        r.w[0] = *reinterpret_cast<const unsigned *>(p);
    } else {
        r.w[0] = *reinterpret_cast<const unsigned short *>(p);
    }
}

// The bfloat16 row widened to float32, with the zero bits taken from a register z (always 0) that the
// caller loads just before the row is used.  The dependency keeps the
// compiler from converting all 32 register-held rows at once, long before
// they are needed (which would triple the registers V occupies).
template <int E>
__device__ __forceinline__ void unpack_row_late(const RawRow<E> &r, unsigned z, float (&f)[E])
{
    unsigned a[E];
#pragma unroll
    for (int k = 0; k < (E + 1) / 2; ++k) {
        // prmt: bytes 0-3 from the row word, bytes 4-7 from z
        asm("prmt.b32 %0, %1, %2, 0x1044;" : "=r"(a[2 * k]) : "r"(r.w[k]), "r"(z));
        if (2 * k + 1 < E) asm("prmt.b32 %0, %1, %2, 0x3244;" : "=r"(a[2 * k + 1]) : "r"(r.w[k]), "r"(z));
    }
#pragma unroll
    for (int e = 0; e < E; ++e) f[e] = __uint_as_float(a[e]);
}

// Non-blocking test of an mbarrier phase by a whole warp: true only when
// every lane has observed the phase complete (each lane then has acquired
// the data released with it).
__device__ __forceinline__ bool warp_test_bar(uint64_t *bar, unsigned parity)
{
    return __all_sync(kFull, ptx::mbar_try_wait(bar, parity));
}

// Combine the four compute warps' aggregates (in shared memory) into the
// chunk's aggregate, in warp order.
template <int D>
__device__ __forceinline__ void chunk_aggregate(const float *wst, float &am,
                                                float (&au)[VLayout<D>::E], float &aw, int lane)
{
    constexpr int E = VLayout<D>::E;
    constexpr int SS = StateLayout<D>::SS;
    read_state_smem<D>(wst, am, au, aw, lane);
#pragma unroll
    for (int k = 1; k < kPipeComputeWarps; ++k) {
        float bm, bw, bu[E];
        read_state_smem<D>(wst + k * SS, bm, bu, bw, lane);
        combine_into<E>(am, au, aw, bm, bu, bw);
        am = bm;
        aw = bw;
#pragma unroll
        for (int e = 0; e < E; ++e) au[e] = bu[e];
    }
}

// Decoupled look-back of chunk c (carry warp) whose fold reads the
// predecessors' states through shared memory.  This kernel keeps the
// chunks' aggregates in one array (states + chunk * SS) and their inclusive
// prefixes in another (states + (chunks + chunk) * SS), so the aggregates of
// consecutive predecessors are contiguous.  A window of 32 predecessors is
// polled as in lookback(); once it resolves, every predecessor but the last
// has only an aggregate, and the last may hold an inclusive prefix.  Lane 0
// then starts at most two 1-D bulk copies per round of up to FOLD states
// (the round's aggregates, in one piece, and the inclusive prefix) into the
// group's fold buffer `fb`, on the mbarrier `fbar`: the states cross from L2
// in one round trip and occupy no registers while in flight.  (A copy per
// state cost more to issue than the round trip; splitting the aggregates
// over several lanes' copies cost more in fences than it gained in landing
// time; folding from registers took a round trip per six states.)  The fold then reads shared memory, in any
// order of the states (one maximum over all of them, then a weighted sum).
// The states are published with release semantics and the flags read with
// acquire by each lane; the warp barrier orders those acquires before lane
// 0's proxy fence and copies.
// `fb_phase` is the parity of the fold barrier's next phase; `fb_busy` stays
// true if a wait for copies gave up (the caller waits for them before the
// block's shared memory can go).  False when a wait gave up or a
// predecessor was poisoned.
template <int D, int FOLD>
__device__ bool lookback_bulk(const ScanParams &p, int64_t head, int64_t c, float &xm,
                              float (&xu)[VLayout<D>::E], float &xw, int lane, float *fb, uint64_t *fbar,
                              unsigned &fb_phase, bool &fb_busy, int64_t wait_limit)
{
    using L = VLayout<D>;
    constexpr int E = L::E;
    constexpr int SS = StateLayout<D>::SS;
    const int64_t first = head * p.chunks_per_head;   // chunk 0 of this head
    const bool owns = (L::LANES == 32 || lane < L::LANES);
    // every predecessor slot read below lies in [first, first + c), inside the workspace
    if (!AAREN_IN_BOUNDS(p.status, c <= p.chunks_per_head && in_range(first, c, p.heads * p.chunks_per_head)))
        return false;
    if (fb_busy) {   // copies of an earlier fold that gave up: let them land first
        if (!wait_bar(fbar, fb_phase, wait_limit)) return false;
        fb_busy = false;
        fb_phase ^= 1u;
    }
    for (int64_t j0 = c - 1; j0 >= 0; j0 -= 32) {
        const int64_t j = j0 - lane;
        const bool has = (j >= 0);   // lanes before chunk 0 act as a stop
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
            __nanosleep(sleep_ns);
            if (sleep_ns < 256) sleep_ns *= 2;
        }
        __syncwarp();   // every lane's acquire before lane 0's copies
        // predecessors 0..k of the window (lanes before chunk 0 are never
        // copied: the first of them is the stop k, an identity).  Predecessor
        // i of the window is chunk j0 - i of the head.
        const int last = (j0 - k >= 0) ? k : static_cast<int>(j0);   // the window's last real predecessor
        const size_t chunks = size_t(p.heads) * size_t(p.chunks_per_head);
        for (int i0 = 0; i0 <= last; i0 += FOLD) {
            const int n = (last + 1 - i0 < FOLD) ? last + 1 - i0 : FOLD;
            // the round covers chunks j0 - i0 - n + 1 .. j0 - i0; only its
            // last predecessor (the lowest chunk) can hold an inclusive prefix
            const unsigned f_end = __shfl_sync(kFull, f, (i0 + n - 1) & 31);
            const int n_inc = (f_end == FLAG_INC) ? 1 : 0;
            const int n_agg = n - n_inc;
            if (lane == 0) {
                const size_t low = size_t(first + (j0 - i0 - n + 1));   // the round's lowest chunk
                ptx::mbar_arrive_expect_tx(fbar, static_cast<unsigned>(n) * SS * sizeof(float));
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // earlier reads of fb first
                ptx::fence_proxy_async_global();
                if (n_agg > 0)
                    ptx::bulk_g2s_plain(fb, p.states + (low + n_inc) * SS,
                                        static_cast<unsigned>(n_agg) * SS * sizeof(float), fbar);
                if (n_inc)
                    ptx::bulk_g2s_plain(fb + n_agg * SS, p.states + (chunks + low) * SS, SS * sizeof(float), fbar);
            }
            fb_busy = true;
            if (!wait_bar(fbar, fb_phase, wait_limit)) return false;
            fb_busy = false;
            fb_phase ^= 1u;
            // fold x := (these states) (+) x: scalars lane-parallel, u per lane over its dims
            float mi = -INFINITY, wi = 0.f;
            if (lane < n) {
                mi = fb[lane * SS];
                wi = fb[lane * SS + 1];
            }
            const float M = fmaxf(warp_max(mi), xm);
            const float ei = (lane < n) ? exp_rel(mi, M) : 0.f;
            float acc[E];
#pragma unroll
            for (int e = 0; e < E; ++e) acc[e] = 0.f;
#pragma unroll 4
            for (int b = 0; b < n; ++b) {
                const float eb = __shfl_sync(kFull, ei, b);
                if (owns) {
                    float v[E];
                    load_vals<E>(fb + b * SS + 4 + lane * E, v);
#pragma unroll
                    for (int e = 0; e < E; ++e) acc[e] = fmaf(eb, v[e], acc[e]);
                }
            }
            const float wsum = warp_sum(ei * wi);
            const float ex = (xm == -INFINITY) ? 0.f : exp_rel(xm, M);
#pragma unroll
            for (int e = 0; e < E; ++e) xu[e] = fmaf(ex, xu[e], acc[e]);
            xw = fmaf(ex, xw, wsum);
            xm = M;
            __syncwarp();   // every lane's reads of fb before the next copies
        }
        if (inc != 0) return true;   // lane k held an inclusive prefix (or the head start)
    }
    return true;
}

#ifndef AAREN_PIPE_SPIN_WAIT
#define AAREN_PIPE_SPIN_WAIT 0
#endif
// How compute warps wait for their stage and their carry.
__device__ __forceinline__ bool compute_wait(uint64_t *bar, unsigned parity, int64_t limit_ns)
{
    return AAREN_PIPE_SPIN_WAIT ? wait_bar_spin(bar, parity, limit_ns) : wait_bar(bar, parity, limit_ns);
}

template <int D, typename Tout, int GROUPS, int STAGES, typename Tin = __nv_bfloat16>
__global__ void __launch_bounds__(PipeTile<D, GROUPS, STAGES, Tin>::THREADS, 1)
    k_scan_pipe(const ScanParams p, const int64_t total_chunks)
{
    using L = VLayout<D>;
    using T = PipeTile<D, GROUPS, STAGES, Tin>;
    constexpr int E = L::E;
    constexpr int C = T::C;
    constexpr int SS = T::SS;
    constexpr int WS = kPipeComputeWarps * SS;   // floats of one set of warp states

    extern __shared__ __align__(128) unsigned char smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = warp / kPipeGroupWarps;        // group
    const int role = warp % kPipeGroupWarps;     // 0..3 compute warp, 4 carry warp
    unsigned char *gs = smem + T::group_off + size_t(g) * T::group_bytes;
    float *wst = reinterpret_cast<float *>(gs + T::g_wst);   // [2][4][SS]
    float *cst = reinterpret_cast<float *>(gs + T::g_cst);   // [4][SS]
    // the group's current chunk: ticket, pool stage, parity of that stage's fill
    volatile long long *meta_t = reinterpret_cast<volatile long long *>(gs + T::g_meta);
    volatile int *meta_s = reinterpret_cast<volatile int *>(gs + T::g_meta + 8);
    volatile int *fail = reinterpret_cast<volatile int *>(gs + T::g_meta + 12);
    uint64_t *gbars = reinterpret_cast<uint64_t *>(gs + T::g_bars);
    uint64_t *metab = gbars + 0;    // the group's next chunk is known (carry warp)
    uint64_t *empty = gbars + 1;    // the chunk's stage has been read (4 compute warps)
    uint64_t *aggb = gbars + 2;     // warp aggregates written (4 compute warps)
    uint64_t *carryb = gbars + 3;   // the chunk's carry written (carry warp)
    uint64_t *cagg = gbars + 4;     // the chunk aggregate written (compute warp 1)
    uint64_t *fbar = gbars + 5;     // look-back states landed in the fold buffer (bulk copies)
    float *fb = reinterpret_cast<float *>(smem + T::fold_off + size_t(g) * T::fold_bytes);
    unsigned *pool = reinterpret_cast<unsigned *>(smem + T::pool_off);          // free stages
    unsigned *fills = reinterpret_cast<unsigned *>(smem + T::fills_off);        // per stage
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + T::full_off);          // per stage
    const bool owns = (L::LANES == 32 || lane < L::LANES);

    if (threadIdx.x == 0) {
        *pool = (STAGES == 32) ? 0xffffffffu : ((1u << STAGES) - 1u);
        for (int st = 0; st < STAGES; ++st) {
            fills[st] = 0;
            ptx::mbar_init(full + st, 1);
        }
    }
    if (role == kPipeComputeWarps && lane == 0) {
        ptx::mbar_init(metab, 1);
        ptx::mbar_init(empty, kPipeComputeWarps);
        ptx::mbar_init(aggb, kPipeComputeWarps);
        ptx::mbar_init(carryb, 1);
        ptx::mbar_init(cagg, 1);
        ptx::mbar_init(fbar, 1);
    }
    if (threadIdx.x == 0) ptx::fence_barrier_init();
    // launched as a programmatic dependent of the workspace zeroing: the set-up
    // above overlaps it, and nothing in global memory is touched before it
    // has completed
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __syncthreads();
    // waits on the group's own barriers may legitimately last as long as a
    // look-back wait, so they get a wider limit
    const int64_t group_limit = p.wait_limit_ns * 16;

    if (role == kPipeComputeWarps) {
        // ------------------------------------------------------------ carry warp
        const uint64_t pol = ptx::policy_evict_first();
        int held = -1;                // stage with a copy this warp issued (its chunk not yet aggregated)
        unsigned held_par = 0;
        unsigned fb_phase = 0;        // parity of the fold barrier's next phase
        bool fb_busy = false;         // fold copies possibly still in flight
        // Claim a free stage of the block's pool, take the group's next
        // ticket and start the chunk's copies; or post a stop.  False when no
        // stage came free in time.
        auto issue = [&]() -> bool {
            long long t = kTicketStop;
            int st = -1;
            unsigned par = 0;
            int ok = 1;
            if (lane == 0) {
                const uint64_t t_start = ptx::globaltimer();
                for (unsigned polls = 0;; ++polls) {
                    const unsigned m = *reinterpret_cast<volatile unsigned *>(pool);
                    if (m != 0) {
                        const int cand = __ffs(m) - 1;
                        if (atomicAnd(pool, ~(1u << cand)) & (1u << cand)) {
                            st = cand;
                            break;
                        }
                        continue;
                    }
                    if (polls >= kMinWaitPolls &&
                        int64_t(ptx::globaltimer() - t_start) > group_limit) {
                        ok = 0;
                        break;
                    }
                    __nanosleep(64);
                }
                if (ok) {
                    __threadfence_block();
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    t = static_cast<long long>(atomicAdd(p.ticket, 1u));
                    if (t >= total_chunks) {
                        t = kTicketStop;
                        atomicOr(pool, 1u << st);   // nothing to load: give the stage back
                        st = -1;
                    }
                    if (st >= 0) {
                        par = fills[st] & 1u;
                        fills[st] = fills[st] + 1;
                    }
                    *meta_t = t;
                    *meta_s = st | static_cast<int>(par << 8);
                    if (t >= 0) {
                        const int64_t c = t / p.heads;
                        const int64_t head = t - c * p.heads;
                        const int64_t t0 = c * C;
                        const int nvalid = static_cast<int>(p.N - t0 < C ? p.N - t0 : C);
                        const unsigned bytes = static_cast<unsigned>(nvalid) * D * sizeof(Tin);
                        const int64_t row0 = head * p.N + t0;
                        unsigned char *stage = smem + size_t(st) * T::stage_bytes;
                        // a stage of the pool, the chunk's rows of K and V and the head's q
                        if (AAREN_IN_BOUNDS(p.status, st < STAGES && nvalid >= 1 && nvalid <= C &&
                                                          in_range(row0, nvalid, p.heads * p.N) &&
                                                          in_range(head, 1, p.heads))) {
                            ptx::mbar_arrive_expect_tx(full + st, 2 * bytes + unsigned(T::q_bytes));
                            ptx::bulk_g2s(stage, static_cast<const Tin *>(p.K) + row0 * D, bytes, full + st,
                                          pol);
                            ptx::bulk_g2s(stage + T::st_v, static_cast<const Tin *>(p.V) + row0 * D, bytes,
                                          full + st, pol);
                            ptx::bulk_g2s(stage + T::st_q, static_cast<const Tin *>(p.q) + head * D,
                                          unsigned(T::q_bytes), full + st, pol);
                        } else if (st < STAGES) {
                            ptx::mbar_arrive(full + st);   // no copy: the fill completes at once
                        }
                    }
                    ptx::mbar_arrive(metab);
                }
            }
            ok = __shfl_sync(kFull, ok, 0);
            t = __shfl_sync(kFull, t, 0);
            st = __shfl_sync(kFull, st, 0);
            par = __shfl_sync(kFull, par, 0);
            if (ok && t >= 0) {
                held = st;
                held_par = par;
            }
            return ok != 0 && t >= 0;
        };

        bool live = issue();
        int64_t it = 0;
        for (; live; ++it) {
            const long long t = __shfl_sync(kFull, lane == 0 ? *meta_t : 0ll, 0);
            const unsigned par = static_cast<unsigned>(it & 1);
            const int64_t c = t / p.heads;
            const int64_t head = t - c * p.heads;
            const int64_t chunk = head * p.chunks_per_head + c;   // workspace slot
            // the chunk's workspace slot and the head's state rows
            const bool slot_ok = AAREN_IN_BOUNDS(p.status, in_range(chunk, 1, p.heads * p.chunks_per_head) &&
                                                               in_range(head, 1, p.heads));
            const bool publish = (chunk != p.fault_chunk) && slot_ok;
            bool issued = false;   // the group's next chunk was already started
            unsigned *my_flag = p.flags + chunk;
            // this chunk's inclusive prefix (its aggregate is at states + chunk * SS)
            float *my_inc = p.states + (size_t(p.heads) * size_t(p.chunks_per_head) + size_t(chunk)) * SS;

            float xm = -INFINITY, xw = 0.f, xu[E];
#pragma unroll
            for (int e = 0; e < E; ++e) xu[e] = 0.f;
            bool lb_ok = true;
            if (c == 0) {
                if (p.m_in != nullptr && slot_ok) {
                    xm = p.m_in[head];
                    xw = p.w_in[head];
                    if (owns) load_vals<E>(p.u_in + head * D + lane * E, xu);
                }
            } else {
                lb_ok = slot_ok && lookback_bulk<D, T::FOLD>(p, head, c, xm, xu, xw, lane, fb, fbar, fb_phase,
                                                             fb_busy, group_limit);
            }
            // the chunk aggregate, formed by compute warp 1 (slot 1 of cst)
            if (!wait_bar(cagg, par, group_limit)) {
                if (lane == 0) atomicOr(p.status, STATUS_LOAD_TIMEOUT);
                break;   // the compute warps stopped
            }
            held = -1;   // the compute warps have consumed the copy
            if (lb_ok) {
                float im, iw, iu[E];
                read_state_smem<D>(cst + SS, im, iu, iw, lane);
                // the carry into the chunk (slot 0): each compute warp adds
                // the aggregates of the warps before it itself, so the carry
                // warp hands over one state and goes on to the inclusive prefix
                write_state<D>(cst, xm, xu, xw, lane);
                if (lane == 0) *fail = 0;
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(carryb);
                // the group's next chunk starts now: what is left of this one
                // (its inclusive prefix) waits on nothing, so its successors
                // are not held up and tickets still finish in order
                live = issue();
                issued = true;
                combine_into<E>(xm, xu, xw, im, iu, iw);   // inclusive = exclusive (+) aggregate
                if (publish) {
                    write_state<D>(my_inc, im, iu, iw, lane);
                    publish_flag(my_flag, FLAG_INC, lane);
                }
                if (c == p.chunks_per_head - 1 && p.m_out != nullptr) {
                    if (lane == 0) {
                        p.m_out[head] = im;
                        p.w_out[head] = iw;
                    }
                    if (owns) store_vals<E>(p.u_out + head * D + lane * E, iu);
                }
            } else {
                if (lane == 0) {
                    if (slot_ok) atomicOr(p.status, STATUS_LOOKBACK_TIMEOUT);
                    *fail = 1;
                }
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(carryb);
                if (publish) publish_flag(my_flag, FLAG_POISON, lane);
            }
            if (!issued) live = issue();
        }
        // A copy this warp issued can still be in flight only if the compute
        // warps stopped early: wait for it before the block's memory goes.
        if (held >= 0 && lane == 0) wait_bar(full + held, held_par, group_limit);
        if (fb_busy && lane == 0) wait_bar(fbar, fb_phase, group_limit);   // fold copies still in flight
        return;
    }

    // ------------------------------------------------------------ compute warps
    const int wg = role;
    float4 *cf = reinterpret_cast<float4 *>(gs + T::g_coef) + wg * 32;
    for (int64_t it = 0;; ++it) {
        const unsigned par = static_cast<unsigned>(it & 1);
        if (!compute_wait(metab, par, group_limit)) {
            if (lane == 0) atomicOr(p.status, STATUS_LOAD_TIMEOUT);
            break;
        }
        const long long t = *meta_t;
        if (t < 0) break;
        const int st_word = *meta_s;
        const int st = st_word & 0xff;
        const unsigned fill_par = static_cast<unsigned>(st_word >> 8) & 1u;
        if (!AAREN_IN_BOUNDS(p.status, st < STAGES)) break;   // a stage of the pool
        if (!compute_wait(full + st, fill_par, group_limit)) {
            if (lane == 0) atomicOr(p.status, STATUS_LOAD_TIMEOUT);
            break;
        }
        const unsigned char *stage = smem + size_t(st) * T::stage_bytes;
        const int64_t c = t / p.heads;
        const int64_t head = t - c * p.heads;
        const int64_t t0 = c * C;
        const int nvalid = static_cast<int>(p.N - t0 < C ? p.N - t0 : C);
        int nv = nvalid - wg * 32;                            // valid rows of this warp
        nv = nv < 0 ? 0 : (nv > 32 ? 32 : nv);
        // this warp's rows of O and stats, and the chunk's workspace slot
        // (on a violation the warp computes but writes nothing)
        // (a warp past the end of a ragged last chunk has no rows: nv = 0)
        const bool rows_ok = AAREN_IN_BOUNDS(
            p.status, (nv == 0 || in_range(head * p.N + t0 + wg * 32, nv, p.heads * p.N)) &&
                          in_range(head * p.chunks_per_head + c, 1, p.heads * p.chunks_per_head));

        // 1. scores, lane = token.  float32 keys: the compensated dot product
        //    of the one-chunk-per-block kernel and the backward pass;
        //    bfloat16 keys: the mixed-precision dot product the backward pass
        //    also uses (the same functions, so every kernel sees bitwise the
        //    same score).
        const Tin *Vw = reinterpret_cast<const Tin *>(stage + T::st_v) + size_t(wg) * 32 * D + lane * E;
        float s = -INFINITY;
        if (lane < nv) {
            const Tin *krow = reinterpret_cast<const Tin *>(stage) + size_t(wg * 32 + lane) * D;
            if constexpr (sizeof(Tin) == 4)
                s = dot_row<D, Tin>(krow, reinterpret_cast<const float *>(stage + T::st_q), lane);
            else
                s = dot_row_bf16<D>(krow, reinterpret_cast<const __nv_bfloat16 *>(stage + T::st_q), lane);
        }
        if (lane >= nv) s = -INFINITY;

        // 2. V rows into registers (for the aggregate and the rescan), then
        //    the warp aggregate (m_w, u_w, w_w), relative to the warp's
        //    maximum, from those registers: the stage is read once for V and
        //    the aggregate, on which every successor's look-back waits, is
        //    out sooner.  Rows past nv are zero and weigh 0.
        PipeRow<Tin, E> vr[32];
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            zero_row<E>(vr[r]);
            if (owns && r < nv) lds_row<E>(Vw + size_t(r) * D, vr[r]);
        }
        const float mw = warp_max(s);
        const float b = (s == -INFINITY) ? 0.f : exp_rel(s, mw);
        const float ww = warp_sum(b);
        {
            // u_w = sum_r b_r v_r over the warp's rows, two dims per packed FMA
            constexpr int P2 = (E + 1) / 2;
            uint64_t u2[P2];
#pragma unroll
            for (int k = 0; k < P2; ++k) u2[k] = 0ull;
            float u1 = 0.f;   // d = 16: one dim per lane
#pragma unroll
            for (int r = 0; r < 32; ++r) {
                const float br = __shfl_sync(kFull, b, r);
                float v[E];
                unpack_row_late<E>(vr[r], 0u, v);
                if constexpr (E >= 2) {
                    const uint64_t bb = pack2(br, br);
#pragma unroll
                    for (int k = 0; k < E / 2; ++k) u2[k] = ffma2(bb, pack2(v[2 * k], v[2 * k + 1]), u2[k]);
                } else {
                    u1 = fmaf(br, v[0], u1);
                }
            }
            float u[E];
            if constexpr (E >= 2) {
#pragma unroll
                for (int k = 0; k < E / 2; ++k) unpack2(u2[k], u[2 * k], u[2 * k + 1]);
            } else {
                u[0] = u1;
            }
            write_state<D>(wst + par * WS + wg * SS, mw, u, ww, lane);
        }
        __syncwarp();
        // (testing hook: warp 0 of one chunk withholds its arrival, so the
        // group's waits on the aggregates give up)
        if (lane == 0 && !(wg == 0 && head * p.chunks_per_head + c == p.drop_chunk))
            ptx::mbar_arrive(aggb);

        // then hand the stage back to the pool (compute warp 0, once all four
        // warps are done with it)
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(empty);
        if (wg == 0) {
            if (lane == 0) {
                if (wait_bar(empty, par, group_limit)) {
                    __threadfence_block();
                    atomicOr(pool, 1u << st);
                } else {
                    atomicOr(p.status, STATUS_LOAD_TIMEOUT);
                }
            }
            __syncwarp();
        }

        // 3. compute warp 1 forms the chunk aggregate as soon as the four
        //    warp aggregates exist (warp 0 is busy handing the stage back;
        //    the wait for the carry would otherwise be idle).  It hands it to
        //    the carry warp (for the inclusive prefix) and publishes it for
        //    successors' look-backs: a successor's look-back waits for the
        //    aggregates of every predecessor still in flight, so this
        //    publication sets the pace of the whole scan.  The carry warp
        //    may already have published the inclusive prefix, which wins.
        if (wg == 1) {
            if (compute_wait(aggb, par, group_limit)) {
                float am, aw, au[E];
                chunk_aggregate<D>(wst + par * WS, am, au, aw, lane);
                write_state<D>(cst + SS, am, au, aw, lane);
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(cagg);
                const int64_t chunk = head * p.chunks_per_head + c;
                if (c > 0 && chunk != p.fault_chunk && rows_ok) {
                    write_state<D>(p.states + size_t(chunk) * SS, am, au, aw, lane);
                    publish_agg_if_none(p.flags + chunk, lane);
                }
            }
        }

        // 4. wait for the chunk's carry
        if (!compute_wait(carryb, par, group_limit)) {
            if (lane == 0) atomicOr(p.status, STATUS_LOAD_TIMEOUT);
            break;
        }
        if (*fail) continue;

        // 5. this warp's carry = the chunk's carry (+) the aggregates of the
        //    warps before it, in warp order; then rescan from it, V from
        //    registers, and write O
        if (nv > 0 && rows_ok) {
            float rm, rw, u[E];
            read_state_smem<D>(cst, rm, u, rw, lane);
#pragma unroll 1
            for (int k = 0; k < wg; ++k) {
                float bm, bw, bu[E];
                read_state_smem<D>(wst + par * WS + k * SS, bm, bu, bw, lane);
                combine_into<E>(rm, u, rw, bm, bu, bw);
                rm = bm;
                rw = bw;
#pragma unroll
                for (int e = 0; e < E; ++e) u[e] = bu[e];
            }
            // scalar recurrences across lanes (lane = token)
            float M = s;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(kFull, M, off);
                if (lane >= off) M = fmaxf(M, y);
            }
            M = fmaxf(M, rm);
            float Mp = __shfl_up_sync(kFull, M, 1);
            if (lane == 0) Mp = rm;
            const float alpha = exp_rel(Mp, M);
            const float beta = (s == -INFINITY) ? 0.f : exp_rel(s, M);
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
            const float rcp = (s == -INFINITY) ? 0.f : __frcp_rn(wt);
            if (p.stats != nullptr && lane < nv)   // this prefix's (m, w), for a backward pass
                p.stats[size_t(head * p.N + t0 + wg * 32) + lane] = make_float2(M, wt);
            cf[lane] = make_float4(alpha, beta, rcp, 0.f);   // .w: the zero for unpack_row_late
            __syncwarp();
            Tout *orow = static_cast<Tout *>(p.O) + size_t(head * p.N + t0 + wg * 32) * D + lane * E;
            // Rows in blocks of kRescanBlock: the block body is unrolled (V
            // stays in registers under static names), the blocks are not, and
            // the register-held rows shift down by one block after each (a
            // few moves, for a loop body that fits the instruction cache).
            // u in packed pairs (two dims per FMA / multiply; d = 16 keeps one)
            constexpr int P2 = (E + 1) / 2;
            uint64_t u2[P2];
            if constexpr (E >= 2) {
#pragma unroll
                for (int k = 0; k < E / 2; ++k) u2[k] = pack2(u[2 * k], u[2 * k + 1]);
            }
#pragma unroll 1
            for (int rb = 0; rb < nv; rb += kRescanBlock) {
#pragma unroll
                for (int i = 0; i < kRescanBlock; ++i) {
                    const int r = rb + i;
                    if (r >= nv) break;
                    const float4 k = cf[r];
                    float v[E], o[E];
                    unpack_row_late<E>(vr[i], __float_as_uint(k.w), v);
                    if constexpr (E >= 2) {
                        if (k.x != 1.0f) {
                            const uint64_t aa = pack2(k.x, k.x);
#pragma unroll
                            for (int j = 0; j < E / 2; ++j) u2[j] = fmul2(u2[j], aa);
                        }
                        const uint64_t bb = pack2(k.y, k.y), rr = pack2(k.z, k.z);
#pragma unroll
                        for (int j = 0; j < E / 2; ++j) {
                            u2[j] = ffma2(bb, pack2(v[2 * j], v[2 * j + 1]), u2[j]);
                            unpack2(fmul2(u2[j], rr), o[2 * j], o[2 * j + 1]);
                        }
                    } else {
                        if (k.x != 1.0f) u[0] *= k.x;
                        u[0] = fmaf(k.y, v[0], u[0]);
                        o[0] = u[0] * k.z;
                    }
                    if (owns) store_vals<E>(orow + size_t(r) * D, o);
                }
#pragma unroll
                for (int i = 0; i + kRescanBlock < 32; ++i) vr[i] = vr[i + kRescanBlock];
            }
            __syncwarp();
        }
    }
}

}  // namespace aaren
