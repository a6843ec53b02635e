// aaren_api.cu -- host side of libaaren: argument checks, tile selection,
// workspace layout, launches and the device status word.  The operation and
// the conventions are documented in include/aaren.h.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstdlib>

#include "aaren.h"
#include "common.cuh"
#include "scan_kernel.cuh"
#include "scan_pipe_kernel.cuh"
#include "reduce_kernel.cuh"
#include "bwd_kernel.cuh"
#include "step_kernel.cuh"
#include "linattn_kernel.cuh"

namespace aaren {

// Per-device status word; kernels OR failure bits into it, aaren_check reads
// and clears it.
__device__ unsigned g_status;

namespace {

constexpr int64_t kDefaultWaitLimitNs = 1000000000;   // 1 s
std::atomic<int64_t> g_fault_chunk{-1};
std::atomic<int64_t> g_drop_chunk{-1};
std::atomic<int64_t> g_bounds_probe{0};
std::atomic<int64_t> g_wait_limit_ns{kDefaultWaitLimitNs};

constexpr size_t kHeaderBytes = 256;   // ticket counter, padded

bool supported_d(int64_t d) { return d == 16 || d == 32 || d == 64 || d == 128; }
bool supported_dtype(int32_t t) { return t == AAREN_F32 || t == AAREN_BF16 || t == AAREN_BF16_F32OUT; }

size_t in_elem_bytes(int32_t dtype) { return dtype == AAREN_F32 ? 4 : 2; }
size_t out_elem_bytes(int32_t dtype) { return dtype == AAREN_BF16 ? 2 : 4; }

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// a * b without int64 overflow (a, b >= 0)
bool mul_ok(int64_t a, int64_t b, int64_t *out)
{
    if (a != 0 && b > INT64_MAX / a) return false;
    *out = a * b;
    return true;
}

// Tile shape per (d, input type): warps per block and 32-token groups per
// warp; a chunk is warps * groups * 32 tokens.  Chosen so K and V of one
// chunk fill about 64 KB of shared memory (3 blocks per SM).
template <int D, typename Tin>
struct TileChoice {
    static constexpr int WARPS = (sizeof(Tin) == 4 && D == 128) ? 2 : 4;
    static constexpr int GROUPS = 1;
    static constexpr int C = WARPS * GROUPS * 32;
};

int64_t chunk_tokens(int64_t d, int32_t dtype)
{
    const bool f32 = (dtype == AAREN_F32);
    switch (d) {
    case 16: return f32 ? TileChoice<16, float>::C : TileChoice<16, __nv_bfloat16>::C;
    case 32: return f32 ? TileChoice<32, float>::C : TileChoice<32, __nv_bfloat16>::C;
    case 64: return f32 ? TileChoice<64, float>::C : TileChoice<64, __nv_bfloat16>::C;
    case 128: return f32 ? TileChoice<128, float>::C : TileChoice<128, __nv_bfloat16>::C;
    default: return 0;
    }
}

struct WorkspaceLayout {
    size_t flags_off, states_off, bytes, zero_bytes;
    int64_t chunks_per_head, total_chunks;
};

// Workspace: [ticket | pad to 256] [flags: u32 per chunk, padded to 256]
// [states: per chunk 2 x (d + 4) floats].  Only the ticket and the flags need
// zeroing before a launch (zero_bytes).
bool workspace_layout(int64_t BH, int64_t N, int64_t d, int64_t C, WorkspaceLayout *w)
{
    if (C <= 0) return false;
    const int64_t cph = (N + C - 1) / C;
    int64_t total;
    if (!mul_ok(BH, cph, &total)) return false;
    if (total > INT_MAX) return false;   // one block per chunk, 32-bit ticket
    w->chunks_per_head = cph;
    w->total_chunks = total;
    const size_t flag_bytes = ((size_t(total) * 4 + 255) / 256) * 256;
    w->flags_off = kHeaderBytes;
    w->states_off = kHeaderBytes + flag_bytes;
    w->zero_bytes = kHeaderBytes + flag_bytes;
    w->bytes = w->states_off + size_t(total) * 2 * size_t(d + 4) * sizeof(float);
    return true;
}

template <typename Kernel>
cudaError_t allow_smem(Kernel kern, size_t bytes, std::atomic<unsigned long long> &done)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (done.load() & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes));
    if (e == cudaSuccess) done.fetch_or(bit);
    return e;
}

// A scan kernel launched as the programmatic dependent of the workspace
// zeroing before it (k_zero_ws): its launch may begin while the zeroing runs;
// the kernel waits for the zeroing's completion before any global access.
template <typename... Args>
cudaError_t launch_dependent(void (*kern)(Args...), unsigned grid, unsigned block, size_t smem,
                             cudaStream_t st, Args... args)
{
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// The ticket and flags of a scan workspace (bytes: a multiple of 16) zeroed
// by k_zero_ws, in plain stream order.
cudaError_t zero_scan_workspace(void *ws, size_t bytes, cudaStream_t st)
{
    const int64_t n16 = int64_t(bytes / 16);
    int64_t blocks = (n16 + 255) / 256;
    if (blocks > 1184) blocks = 1184;
    if (blocks < 1) blocks = 1;
    k_zero_ws<<<unsigned(blocks), 256, 0, st>>>(static_cast<uint4 *>(ws), n16);
    return cudaGetLastError();
}

template <int D, typename Tin, typename Tout>
aaren_status_t launch_scan(const ScanParams &p, int64_t total_chunks, cudaStream_t st)
{
    using TC = TileChoice<D, Tin>;
    using Tile = ScanTile<D, Tin, TC::WARPS, TC::GROUPS>;
    static std::atomic<unsigned long long> configured{0};
    auto kern = k_scan_fwd<D, Tin, Tout, TC::WARPS, TC::GROUPS>;
    if (allow_smem(kern, Tile::smem_bytes, configured) != cudaSuccess) return AAREN_ERR_CUDA;
    return launch_dependent(kern, unsigned(total_chunks), TC::WARPS * 32, Tile::smem_bytes, st, p) == cudaSuccess
               ? AAREN_OK
               : AAREN_ERR_CUDA;
}

// Shape of the persistent bfloat16 kernel per d: groups (five warps each,
// one 128-token chunk in flight) and stages in the block's pool (K, V and q
// of one chunk each; 64 KB at d = 128).  A group holds a stage only from its
// copy until its V rows are in registers, about a quarter of a chunk's
// life, so fewer stages than groups suffice: at d = 128 two (measured as
// fast as three), which leaves room for the groups' look-back fold buffers.
#ifndef AAREN_PIPE_GROUPS_D128
#define AAREN_PIPE_GROUPS_D128 4
#endif
#ifndef AAREN_PIPE_STAGES_D128
#define AAREN_PIPE_STAGES_D128 2
#endif
#ifndef AAREN_PIPE_STAGES_F32_D64
#define AAREN_PIPE_STAGES_F32_D64 3
#endif
#ifndef AAREN_PIPE_GROUPS_D64
#define AAREN_PIPE_GROUPS_D64 4
#endif
#ifndef AAREN_PIPE_STAGES_D64
#define AAREN_PIPE_STAGES_D64 4
#endif
template <int D, typename Tin = __nv_bfloat16>
struct PipeChoice {
    // float32 at d = 64 has the stage size of bfloat16 at d = 128 (64 KB)
    static constexpr int DE = (sizeof(Tin) == 4) ? 2 * D : D;
    static constexpr int GROUPS = (DE == 128) ? AAREN_PIPE_GROUPS_D128 : (DE == 64 ? AAREN_PIPE_GROUPS_D64 : 4);
    static constexpr int STAGES = (sizeof(Tin) == 4 && D == 64) ? AAREN_PIPE_STAGES_F32_D64
                                  : (DE == 128) ? AAREN_PIPE_STAGES_D128 : (DE == 64 ? AAREN_PIPE_STAGES_D64 : 4);
};

int sm_count()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

template <int D, typename Tout, typename Tin = __nv_bfloat16>
aaren_status_t launch_pipe(const ScanParams &p, int64_t total_chunks, cudaStream_t st)
{
    using PC = PipeChoice<D, Tin>;
    using Tile = PipeTile<D, PC::GROUPS, PC::STAGES, Tin>;
    static std::atomic<unsigned long long> configured{0};
    auto kern = k_scan_pipe<D, Tout, PC::GROUPS, PC::STAGES, Tin>;
    if (allow_smem(kern, Tile::smem_bytes, configured) != cudaSuccess) return AAREN_ERR_CUDA;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, Tile::THREADS,
                                                      Tile::smem_bytes) != cudaSuccess ||
        per_sm < 1)
        return AAREN_ERR_CUDA;
    const int sms = sm_count();
    if (sms <= 0) return AAREN_ERR_CUDA;
    int64_t grid = int64_t(sms) * per_sm;
    if (grid > total_chunks) grid = total_chunks;
    return launch_dependent(kern, unsigned(grid), Tile::THREADS, Tile::smem_bytes, st, p, total_chunks) ==
                   cudaSuccess
               ? AAREN_OK
               : AAREN_ERR_CUDA;
}

template <int D>
aaren_status_t dispatch_scan_dtype(const ScanParams &p, int64_t total, int32_t dtype,
                                   cudaStream_t st)
{
    switch (dtype) {
    case AAREN_F32:
        // float32 d = 64 (a 64 KB stage, as bfloat16 at d = 128) runs on the
        // persistent kernel; other float32 sizes on the one-chunk-per-block one
        if constexpr (D == 64) return launch_pipe<D, float, float>(p, total, st);
        else return launch_scan<D, float, float>(p, total, st);
#ifdef AAREN_BF16_BLOCK_KERNEL
    case AAREN_BF16: return launch_scan<D, __nv_bfloat16, __nv_bfloat16>(p, total, st);
    case AAREN_BF16_F32OUT: return launch_scan<D, __nv_bfloat16, float>(p, total, st);
#else
    case AAREN_BF16: return launch_pipe<D, __nv_bfloat16>(p, total, st);
    case AAREN_BF16_F32OUT: return launch_pipe<D, float>(p, total, st);
#endif
    default: return AAREN_ERR_UNSUPPORTED;
    }
}

aaren_status_t dispatch_scan(const ScanParams &p, int64_t total, int64_t d, int32_t dtype,
                             cudaStream_t st)
{
    switch (d) {
    case 16: return dispatch_scan_dtype<16>(p, total, dtype, st);
    case 32: return dispatch_scan_dtype<32>(p, total, dtype, st);
    case 64: return dispatch_scan_dtype<64>(p, total, dtype, st);
    case 128: return dispatch_scan_dtype<128>(p, total, dtype, st);
    default: return AAREN_ERR_UNSUPPORTED;
    }
}

template <int D, typename Tin, typename Tout>
aaren_status_t launch_step(const StepParams &p, cudaStream_t st)
{
    const int64_t threads = p.n * 32;
    // programmatic stream serialisation: the step may begin launching while
    // the kernel before it finishes; k_step waits for that kernel's completion
    // (griddepcontrol.wait) before it reads anything
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned((threads + 255) / 256));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_step<D, Tin, Tout>, p) == cudaSuccess ? AAREN_OK : AAREN_ERR_CUDA;
}

template <int D>
aaren_status_t dispatch_step_dtype(const StepParams &p, int32_t dtype, cudaStream_t st)
{
    switch (dtype) {
    case AAREN_F32: return launch_step<D, float, float>(p, st);
    case AAREN_BF16: return launch_step<D, __nv_bfloat16, __nv_bfloat16>(p, st);
    case AAREN_BF16_F32OUT: return launch_step<D, __nv_bfloat16, float>(p, st);
    default: return AAREN_ERR_UNSUPPORTED;
    }
}

aaren_status_t launch_state_init(float *m, float *u, float *w, int64_t n, int64_t d,
                                 cudaStream_t st)
{
    const int64_t total = n * d;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    k_state_init<<<unsigned(blocks), 256, 0, st>>>(m, u, w, n, d);
    return cudaGetLastError() == cudaSuccess ? AAREN_OK : AAREN_ERR_CUDA;
}

bool overlaps(const void *a, size_t abytes, const void *b, size_t bbytes)
{
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bbytes && b0 < a0 + abytes;
}

// The state triple must be all NULL or all set; u 16-byte, m and w 4-byte aligned.
aaren_status_t check_state(const float *m, const float *u, const float *w)
{
    const int set = (m != nullptr) + (u != nullptr) + (w != nullptr);
    if (set != 0 && set != 3) return AAREN_ERR_INVALID;
    if (set == 3 && (!aligned(u, 16) || !aligned(m, 4) || !aligned(w, 4))) return AAREN_ERR_INVALID;
    return AAREN_OK;
}

// ---------------------------------------------------------------- backward

int64_t bwd_chunk_tokens(int64_t d, int32_t dtype)
{
    switch (d) {
#define AAREN_BWD_C(DD)                                                                          \
    case DD:                                                                                     \
        return dtype == AAREN_F32 ? BwdTile<DD, float, float>::C                                 \
               : dtype == AAREN_BF16 ? BwdTile<DD, __nv_bfloat16, __nv_bfloat16>::C              \
                                     : BwdTile<DD, __nv_bfloat16, float>::C;
        AAREN_BWD_C(16)
        AAREN_BWD_C(32)
        AAREN_BWD_C(64)
        AAREN_BWD_C(128)
#undef AAREN_BWD_C
    default: return 0;
    }
}

struct BwdLayout {
    size_t flags_off, states_off, acc_off, count_off, bytes, zero_from, zero_bytes;
    int64_t chunks_per_head, total_chunks;
};

// [ticket | pad 256] [flags] [states: 2 per chunk] [dq accumulator: heads x d
// floats] [dq counters: heads]; the ticket, flags, accumulator and counters
// are zeroed before a launch (two ranges).
bool bwd_layout(int64_t BH, int64_t N, int64_t d, int64_t C, BwdLayout *w)
{
    if (C <= 0) return false;
    const int64_t cph = (N + C - 1) / C;
    int64_t total;
    if (!mul_ok(BH, cph, &total) || total > INT_MAX) return false;
    w->chunks_per_head = cph;
    w->total_chunks = total;
    const size_t flag_bytes = ((size_t(total) * 4 + 255) / 256) * 256;
    w->flags_off = kHeaderBytes;
    w->states_off = kHeaderBytes + flag_bytes;
    w->acc_off = w->states_off + size_t(total) * 2 * size_t(d + 4) * sizeof(float);
    w->count_off = w->acc_off + ((size_t(BH) * d * 4 + 255) / 256) * 256;
    w->bytes = w->count_off + ((size_t(BH) * 4 + 255) / 256) * 256;
    w->zero_from = w->acc_off;
    w->zero_bytes = kHeaderBytes + flag_bytes;   // first range; the second is [acc_off, bytes)
    return true;
}

template <int D, typename Tin, typename Tout>
aaren_status_t launch_bwd(const BwdParams &p, int64_t total, cudaStream_t st)
{
    using Tile = BwdTile<D, Tin, Tout>;
    static std::atomic<unsigned long long> configured{0};
    auto kern = k_scan_bwd<D, Tin, Tout>;
    if (allow_smem(kern, Tile::smem_bytes, configured) != cudaSuccess) return AAREN_ERR_CUDA;
    kern<<<unsigned(total), Tile::WARPS * 32, Tile::smem_bytes, st>>>(p);
    return cudaGetLastError() == cudaSuccess ? AAREN_OK : AAREN_ERR_CUDA;
}

template <int D>
aaren_status_t dispatch_bwd_dtype(const BwdParams &p, int64_t total, int32_t dtype, cudaStream_t st)
{
    switch (dtype) {
    case AAREN_F32: return launch_bwd<D, float, float>(p, total, st);
    case AAREN_BF16: return launch_bwd<D, __nv_bfloat16, __nv_bfloat16>(p, total, st);
    case AAREN_BF16_F32OUT: return launch_bwd<D, __nv_bfloat16, float>(p, total, st);
    default: return AAREN_ERR_UNSUPPORTED;
    }
}

aaren_status_t dispatch_bwd(const BwdParams &p, int64_t total, int64_t d, int32_t dtype, cudaStream_t st)
{
    switch (d) {
    case 16: return dispatch_bwd_dtype<16>(p, total, dtype, st);
    case 32: return dispatch_bwd_dtype<32>(p, total, dtype, st);
    case 64: return dispatch_bwd_dtype<64>(p, total, dtype, st);
    case 128: return dispatch_bwd_dtype<128>(p, total, dtype, st);
    default: return AAREN_ERR_UNSUPPORTED;
    }
}

// ---------------------------------------------------------------- reduce

// Parts per head the workspace is sized for: at most 8192 part states in
// all and at least kReduceMinSeg tokens per part.
int64_t reduce_parts_max(int64_t BH, int64_t N)
{
    int64_t by_n = (N + kReduceMinSeg - 1) / kReduceMinSeg;
    int64_t by_total = 8192 / (BH > 0 ? BH : 1);
    int64_t P = by_n < by_total ? by_n : by_total;
    return P < 1 ? 1 : P;
}

struct ReduceLayout {
    size_t parts_off, bytes, zero_bytes;
    int64_t P_max;
};

bool reduce_layout(int64_t BH, int64_t N, int64_t d, ReduceLayout *r)
{
    r->P_max = reduce_parts_max(BH, N);
    int64_t states;
    if (!mul_ok(BH, r->P_max, &states)) return false;
    const size_t counts = ((size_t(BH) * 4 + 255) / 256) * 256;
    r->parts_off = counts;
    r->zero_bytes = counts;
    r->bytes = counts + size_t(states) * size_t(d + 4) * sizeof(float);
    return true;
}

template <int D, typename Tin, typename Tout>
aaren_status_t launch_reduce(ReduceParams p, int64_t P_max, cudaStream_t st)
{
    auto kern = k_scan_reduce<D, Tin, Tout>;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kReduceWarps * 32, 0) != cudaSuccess ||
        per_sm < 1)
        return AAREN_ERR_CUDA;
    const int sms = sm_count();
    if (sms <= 0) return AAREN_ERR_CUDA;
    // one part per resident warp across the GPU (one wave), parts of equal length
    const int64_t target = int64_t(sms) * per_sm * kReduceWarps;
    int64_t P = (target + p.heads - 1) / p.heads;
    if (P > P_max) P = P_max;
    if (P < 1) P = 1;
    int64_t seg = (p.N + P - 1) / P;
    seg = ((seg + kReduceRows - 1) / kReduceRows) * kReduceRows;
    if (seg < kReduceRows) seg = kReduceRows;
    P = (p.N + seg - 1) / seg;
    if (P < 1) P = 1;
    p.P = P;
    p.seg = seg;
    const int64_t warps = p.heads * P;
    const int64_t blocks = (warps + kReduceWarps - 1) / kReduceWarps;
    if (blocks > INT_MAX) return AAREN_ERR_INVALID;
    kern<<<unsigned(blocks), kReduceWarps * 32, 0, st>>>(p);
    return cudaGetLastError() == cudaSuccess ? AAREN_OK : AAREN_ERR_CUDA;
}

template <int D>
aaren_status_t dispatch_reduce_dtype(const ReduceParams &p, int64_t P_max, int32_t dtype, cudaStream_t st)
{
    switch (dtype) {
    case AAREN_F32: return launch_reduce<D, float, float>(p, P_max, st);
    case AAREN_BF16: return launch_reduce<D, __nv_bfloat16, __nv_bfloat16>(p, P_max, st);
    case AAREN_BF16_F32OUT: return launch_reduce<D, __nv_bfloat16, float>(p, P_max, st);
    default: return AAREN_ERR_UNSUPPORTED;
    }
}

aaren_status_t dispatch_reduce(const ReduceParams &p, int64_t P_max, int64_t d, int32_t dtype,
                               cudaStream_t st)
{
    switch (d) {
    case 16: return dispatch_reduce_dtype<16>(p, P_max, dtype, st);
    case 32: return dispatch_reduce_dtype<32>(p, P_max, dtype, st);
    case 64: return dispatch_reduce_dtype<64>(p, P_max, dtype, st);
    case 128: return dispatch_reduce_dtype<128>(p, P_max, dtype, st);
    default: return AAREN_ERR_UNSUPPORTED;
    }
}

// ---- causal cos-re-weighted linear attention -------------------------------

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once through the runtime.
EncodeTiledFn encode_tiled()
{
    static const EncodeTiledFn fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<EncodeTiledFn>(nullptr);
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}

// [BH, N, 64] bfloat16 viewed as a 3-D tensor; boxes of 128 tokens x 64,
// 128-byte swizzle, rows past N read as zero.
bool linattn_map(CUtensorMap *m, const void *base, int64_t BH, int64_t N)
{
    const EncodeTiledFn enc = encode_tiled();
    if (enc == nullptr) return false;
    const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
    const cuuint64_t strides[2] = {64 * 2, static_cast<cuuint64_t>(N) * 64 * 2};
    const cuuint32_t box[3] = {64, la::C, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static_assert(la::kSmemBytes <= 232448, "linear-attention tile exceeds the opt-in shared memory of a CTA");

template <typename Tout>
aaren_status_t launch_linattn(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                              const la::Params &p, cudaStream_t st)
{
    static std::atomic<unsigned long long> configured{0};   // per device
    if (allow_smem(la::k_linattn<Tout>, la::kSmemBytes, configured) != cudaSuccess) return AAREN_ERR_CUDA;
    const int sms = sm_count();
    if (sms <= 0) return AAREN_ERR_CUDA;
    const int64_t grid = p.BH < sms ? p.BH : sms;   // persistent: one CTA per SM, heads strided over them
    la::k_linattn<Tout><<<static_cast<unsigned>(grid), la::kThreads, la::kSmemBytes, st>>>(tq, tk, tv, p);
    return cudaGetLastError() == cudaSuccess ? AAREN_OK : AAREN_ERR_CUDA;
}

}  // namespace
}  // namespace aaren

using namespace aaren;

extern "C" {

aaren_status_t aaren_linattn_forward(const void *Q, const void *K, const void *V, void *O, int64_t B,
                                     int64_t H, int64_t N, int64_t d, double M, int64_t pos0,
                                     int32_t dtype, const float *S_in, const float *z_in, float *S_out,
                                     float *z_out, void *stream)
{
    if (B < 0 || H < 0 || N < 0 || d <= 0 || pos0 < 0) return AAREN_ERR_INVALID;
    if (!(M > 0.0) || !std::isfinite(M)) return AAREN_ERR_INVALID;
    if ((S_in == nullptr) != (z_in == nullptr) || (S_out == nullptr) != (z_out == nullptr))
        return AAREN_ERR_INVALID;
    if (d != la::D) return AAREN_ERR_UNSUPPORTED;
    if (dtype != AAREN_BF16 && dtype != AAREN_BF16_F32OUT) return AAREN_ERR_UNSUPPORTED;
    int64_t BH, tok, elems;
    if (!mul_ok(B, H, &BH) || !mul_ok(BH, N, &tok) || !mul_ok(tok, d, &elems)) return AAREN_ERR_INVALID;
    if (N > INT32_MAX - la::C || BH > INT32_MAX) return AAREN_ERR_INVALID;   // TMA coordinates are 32-bit
    if (S_in != nullptr && (!aligned(S_in, 16) || !aligned(z_in, 4))) return AAREN_ERR_INVALID;
    if (S_out != nullptr && (!aligned(S_out, 16) || !aligned(z_out, 4))) return AAREN_ERR_INVALID;
    if (BH == 0) return AAREN_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t s_bytes = size_t(BH) * 2 * 64 * 64 * sizeof(float), z_bytes = size_t(BH) * 2 * 64 * sizeof(float);
    if (N == 0) {   // nothing to scan: the final state is the starting state
        if (S_out == nullptr) return AAREN_OK;
        const bool ok = (S_in != nullptr)
                            ? cudaMemcpyAsync(S_out, S_in, s_bytes, cudaMemcpyDeviceToDevice, st) == cudaSuccess &&
                                  cudaMemcpyAsync(z_out, z_in, z_bytes, cudaMemcpyDeviceToDevice, st) == cudaSuccess
                            : cudaMemsetAsync(S_out, 0, s_bytes, st) == cudaSuccess &&
                                  cudaMemsetAsync(z_out, 0, z_bytes, st) == cudaSuccess;
        return ok ? AAREN_OK : AAREN_ERR_CUDA;
    }
    if (Q == nullptr || K == nullptr || V == nullptr || O == nullptr) return AAREN_ERR_INVALID;
    if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16)) return AAREN_ERR_INVALID;
    const size_t in_b = size_t(elems) * 2, out_b = size_t(elems) * out_elem_bytes(dtype);
    if (overlaps(O, out_b, Q, in_b) || overlaps(O, out_b, K, in_b) || overlaps(O, out_b, V, in_b))
        return AAREN_ERR_INVALID;
    CUtensorMap tq, tk, tv;
    if (!linattn_map(&tq, Q, BH, N) || !linattn_map(&tk, K, BH, N) || !linattn_map(&tv, V, BH, N))
        return AAREN_ERR_CUDA;
    unsigned *status = nullptr;
    if (cudaGetSymbolAddress(reinterpret_cast<void **>(&status), g_status) != cudaSuccess) return AAREN_ERR_CUDA;
    la::Params p;
    p.O = O;
    p.S_in = S_in; p.z_in = z_in; p.S_out = S_out; p.z_out = z_out;
    p.BH = BH; p.N = N; p.pos0 = pos0;
    p.inv_2M = 1.0 / (2.0 * M);
    p.inv_2Mf = static_cast<float>(p.inv_2M);
    p.status = status;
    p.wait_limit_ns = g_wait_limit_ns.load();
    p.drop_chunk = g_drop_chunk.load();
    return dtype == AAREN_BF16 ? launch_linattn<__nv_bfloat16>(tq, tk, tv, p, st)
                               : launch_linattn<float>(tq, tk, tv, p, st);
}

size_t aaren_scan_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t d)
{
    if (!supported_d(d) || B < 0 || H < 0 || N < 0) return SIZE_MAX;
    int64_t BH;
    if (!mul_ok(B, H, &BH)) return SIZE_MAX;
    if (BH == 0 || N == 0) return 0;
    // the workspace depends on the chunk, which depends on the dtype only for
    // float32 d = 128; take the smaller chunk so the size covers every dtype
    int64_t C = chunk_tokens(d, AAREN_F32);
    const int64_t Cb = chunk_tokens(d, AAREN_BF16);
    if (Cb < C) C = Cb;
    WorkspaceLayout w;
    if (!workspace_layout(BH, N, d, C, &w)) return SIZE_MAX;
    return w.bytes;
}

static aaren_status_t scan_forward_impl(const void *q, const void *K, const void *V, void *O,
                                        int64_t B, int64_t H, int64_t N, int64_t d, int32_t dtype,
                                        const float *m_in, const float *u_in, const float *w_in,
                                        float *m_out, float *u_out, float *w_out, float *stats,
                                        void *workspace, size_t workspace_bytes, void *stream)
{
    if (!supported_dtype(dtype) || !supported_d(d)) return AAREN_ERR_UNSUPPORTED;
    if (B < 0 || H < 0 || N < 0) return AAREN_ERR_INVALID;
    if (check_state(m_in, u_in, w_in) != AAREN_OK) return AAREN_ERR_INVALID;
    if (check_state(m_out, u_out, w_out) != AAREN_OK) return AAREN_ERR_INVALID;
    int64_t BH, BHN, elems;
    if (!mul_ok(B, H, &BH) || !mul_ok(BH, N, &BHN) || !mul_ok(BHN, d, &elems)) return AAREN_ERR_INVALID;
    int64_t kv_bytes, o_bytes;
    if (!mul_ok(elems, int64_t(in_elem_bytes(dtype)), &kv_bytes) ||
        !mul_ok(elems, int64_t(out_elem_bytes(dtype)), &o_bytes))
        return AAREN_ERR_INVALID;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (BH == 0) return AAREN_OK;
    if (N == 0) {
        // final state = starting state
        if (m_out == nullptr) return AAREN_OK;
        if (m_in == nullptr) return launch_state_init(m_out, u_out, w_out, BH, d, st);
        if (cudaMemcpyAsync(m_out, m_in, size_t(BH) * 4, cudaMemcpyDeviceToDevice, st) != cudaSuccess ||
            cudaMemcpyAsync(w_out, w_in, size_t(BH) * 4, cudaMemcpyDeviceToDevice, st) != cudaSuccess ||
            cudaMemcpyAsync(u_out, u_in, size_t(BH) * d * 4, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
            return AAREN_ERR_CUDA;
        return AAREN_OK;
    }
    if (q == nullptr || K == nullptr || V == nullptr || O == nullptr) return AAREN_ERR_INVALID;
    if (!aligned(q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16)) return AAREN_ERR_INVALID;
    if (overlaps(O, size_t(o_bytes), K, size_t(kv_bytes)) || overlaps(O, size_t(o_bytes), V, size_t(kv_bytes)))
        return AAREN_ERR_INVALID;

    const int64_t C = chunk_tokens(d, dtype);
    WorkspaceLayout wl;
    if (!workspace_layout(BH, N, d, C, &wl)) return AAREN_ERR_INVALID;

    void *ws = workspace;
    bool owned = false;
    if (ws == nullptr) {
        if (cudaMallocAsync(&ws, wl.bytes, st) != cudaSuccess) return AAREN_ERR_CUDA;
        owned = true;
    } else if (workspace_bytes < wl.bytes || !aligned(ws, 256)) {
        return AAREN_ERR_WORKSPACE;
    }
    aaren_status_t rc = AAREN_OK;
    if (zero_scan_workspace(ws, wl.zero_bytes, st) != cudaSuccess) {
        rc = AAREN_ERR_CUDA;
    } else {
        unsigned *status = nullptr;
        if (cudaGetSymbolAddress(reinterpret_cast<void **>(&status), g_status) != cudaSuccess) {
            rc = AAREN_ERR_CUDA;
        } else {
            char *base = static_cast<char *>(ws);
            ScanParams p;
            p.q = q; p.K = K; p.V = V; p.O = O;
            p.m_in = m_in; p.u_in = u_in; p.w_in = w_in;
            p.m_out = m_out; p.u_out = u_out; p.w_out = w_out;
            p.ticket = reinterpret_cast<unsigned *>(base);
            p.flags = reinterpret_cast<unsigned *>(base + wl.flags_off);
            p.states = reinterpret_cast<float *>(base + wl.states_off);
            p.status = status;
            p.stats = reinterpret_cast<float2 *>(stats);
            p.N = N;
            p.heads = BH;
            p.chunks_per_head = wl.chunks_per_head;
            p.fault_chunk = g_fault_chunk.load();
            p.drop_chunk = g_drop_chunk.load();
            p.wait_limit_ns = g_wait_limit_ns.load();
            rc = dispatch_scan(p, wl.total_chunks, d, dtype, st);
        }
    }
    if (owned && cudaFreeAsync(ws, st) != cudaSuccess && rc == AAREN_OK) rc = AAREN_ERR_CUDA;
    return rc;
}

size_t aaren_backward_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t d)
{
    if (!supported_d(d) || B < 0 || H < 0 || N < 0) return SIZE_MAX;
    int64_t BH;
    if (!mul_ok(B, H, &BH)) return SIZE_MAX;
    if (BH == 0 || N == 0) return 0;
    int64_t C = bwd_chunk_tokens(d, AAREN_F32);   // the smallest chunk of any dtype
    for (int32_t t : {AAREN_BF16, AAREN_BF16_F32OUT}) {
        const int64_t c = bwd_chunk_tokens(d, t);
        if (c < C) C = c;
    }
    BwdLayout w;
    if (!bwd_layout(BH, N, d, C, &w)) return SIZE_MAX;
    return w.bytes;
}

aaren_status_t aaren_scan_backward(const void *q, const void *K, const void *V, const void *O,
                                   const void *dO, const float *stats, float *dq, float *dK, float *dV,
                                   int64_t B, int64_t H, int64_t N, int64_t d, int32_t dtype,
                                   void *workspace, size_t workspace_bytes, void *stream)
{
    if (!supported_dtype(dtype) || !supported_d(d)) return AAREN_ERR_UNSUPPORTED;
    if (B < 0 || H < 0 || N < 0) return AAREN_ERR_INVALID;
    int64_t BH, BHN, elems;
    if (!mul_ok(B, H, &BH) || !mul_ok(BH, N, &BHN) || !mul_ok(BHN, d, &elems)) return AAREN_ERR_INVALID;
    int64_t in_b, out_b, grad_b;
    if (!mul_ok(elems, int64_t(in_elem_bytes(dtype)), &in_b) ||
        !mul_ok(elems, int64_t(out_elem_bytes(dtype)), &out_b) || !mul_ok(elems, 4, &grad_b))
        return AAREN_ERR_INVALID;
    if (BH == 0) return AAREN_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (dq == nullptr || !aligned(dq, 16)) return AAREN_ERR_INVALID;
    if (N == 0)   // nothing depends on q: its gradient is zero
        return cudaMemsetAsync(dq, 0, size_t(BH) * d * sizeof(float), st) == cudaSuccess
                   ? AAREN_OK : AAREN_ERR_CUDA;
    const void *ins[] = {q, K, V, O, dO, stats, dK, dV};
    for (const void *x : ins)
        if (x == nullptr || !aligned(x, 16)) return AAREN_ERR_INVALID;
    // the gradients must not overlap any input
    const void *rd[] = {K, V, O, dO};
    const size_t rd_b[] = {size_t(in_b), size_t(in_b), size_t(out_b), size_t(out_b)};
    for (int i = 0; i < 4; ++i)
        if (overlaps(dK, size_t(grad_b), rd[i], rd_b[i]) || overlaps(dV, size_t(grad_b), rd[i], rd_b[i]))
            return AAREN_ERR_INVALID;
    if (overlaps(dK, size_t(grad_b), dV, size_t(grad_b))) return AAREN_ERR_INVALID;

    const int64_t C = bwd_chunk_tokens(d, dtype);
    BwdLayout wl;
    if (!bwd_layout(BH, N, d, C, &wl)) return AAREN_ERR_INVALID;
    void *ws = workspace;
    bool owned = false;
    if (ws == nullptr) {
        if (cudaMallocAsync(&ws, wl.bytes, st) != cudaSuccess) return AAREN_ERR_CUDA;
        owned = true;
    } else if (workspace_bytes < wl.bytes || !aligned(ws, 256)) {
        return AAREN_ERR_WORKSPACE;
    }
    aaren_status_t rc = AAREN_OK;
    char *base = static_cast<char *>(ws);
    if (cudaMemsetAsync(base, 0, wl.zero_bytes, st) != cudaSuccess ||
        cudaMemsetAsync(base + wl.zero_from, 0, wl.bytes - wl.zero_from, st) != cudaSuccess) {
        rc = AAREN_ERR_CUDA;
    } else {
        unsigned *status = nullptr;
        if (cudaGetSymbolAddress(reinterpret_cast<void **>(&status), g_status) != cudaSuccess) {
            rc = AAREN_ERR_CUDA;
        } else {
            BwdParams p;
            p.q = q; p.K = K; p.V = V; p.O = O; p.dO = dO;
            p.stats = reinterpret_cast<const float2 *>(stats);
            p.dq = dq; p.dK = dK; p.dV = dV;
            p.ticket = reinterpret_cast<unsigned *>(base);
            p.flags = reinterpret_cast<unsigned *>(base + wl.flags_off);
            p.states = reinterpret_cast<float *>(base + wl.states_off);
            p.dq_acc = reinterpret_cast<float *>(base + wl.acc_off);
            p.dq_count = reinterpret_cast<unsigned *>(base + wl.count_off);
            p.status = status;
            p.N = N;
            p.heads = BH;
            p.chunks_per_head = wl.chunks_per_head;
            p.fault_chunk = g_fault_chunk.load();
            p.wait_limit_ns = g_wait_limit_ns.load();
            rc = dispatch_bwd(p, wl.total_chunks, d, dtype, st);
        }
    }
    if (owned && cudaFreeAsync(ws, st) != cudaSuccess && rc == AAREN_OK) rc = AAREN_ERR_CUDA;
    return rc;
}

size_t aaren_reduce_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t d)
{
    if (!supported_d(d) || B < 0 || H < 0 || N < 0) return SIZE_MAX;
    int64_t BH;
    if (!mul_ok(B, H, &BH)) return SIZE_MAX;
    if (BH == 0) return 0;
    ReduceLayout r;
    if (!reduce_layout(BH, N, d, &r)) return SIZE_MAX;
    return r.bytes;
}

aaren_status_t aaren_scan_reduce(const void *q, const void *K, const void *V, void *o_last, int64_t B,
                                 int64_t H, int64_t N, int64_t d, int32_t dtype, const float *m_in,
                                 const float *u_in, const float *w_in, float *m_out, float *u_out,
                                 float *w_out, void *workspace, size_t workspace_bytes, void *stream)
{
    if (!supported_dtype(dtype) || !supported_d(d)) return AAREN_ERR_UNSUPPORTED;
    if (B < 0 || H < 0 || N < 0) return AAREN_ERR_INVALID;
    if (check_state(m_in, u_in, w_in) != AAREN_OK) return AAREN_ERR_INVALID;
    if (check_state(m_out, u_out, w_out) != AAREN_OK) return AAREN_ERR_INVALID;
    int64_t BH, BHN, elems;
    if (!mul_ok(B, H, &BH) || !mul_ok(BH, N, &BHN) || !mul_ok(BHN, d, &elems)) return AAREN_ERR_INVALID;
    int64_t kv_bytes;
    if (!mul_ok(elems, int64_t(in_elem_bytes(dtype)), &kv_bytes)) return AAREN_ERR_INVALID;
    if (o_last == nullptr && m_out == nullptr) return AAREN_ERR_INVALID;   // nothing to compute
    if (BH == 0) return AAREN_OK;
    // o_N of an empty prefix is 0/0: it needs a starting state
    if (N == 0 && o_last != nullptr && m_in == nullptr) return AAREN_ERR_INVALID;
    if (q == nullptr || (N > 0 && (K == nullptr || V == nullptr))) return AAREN_ERR_INVALID;
    if (!aligned(q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(o_last, 16))
        return AAREN_ERR_INVALID;
    if (o_last != nullptr && (overlaps(o_last, size_t(BH) * d * out_elem_bytes(dtype), K, size_t(kv_bytes)) ||
                              overlaps(o_last, size_t(BH) * d * out_elem_bytes(dtype), V, size_t(kv_bytes))))
        return AAREN_ERR_INVALID;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    ReduceLayout rl;
    if (!reduce_layout(BH, N, d, &rl)) return AAREN_ERR_INVALID;
    void *ws = workspace;
    bool owned = false;
    if (ws == nullptr) {
        if (cudaMallocAsync(&ws, rl.bytes, st) != cudaSuccess) return AAREN_ERR_CUDA;
        owned = true;
    } else if (workspace_bytes < rl.bytes || !aligned(ws, 256)) {
        return AAREN_ERR_WORKSPACE;
    }
    aaren_status_t rc = AAREN_OK;
    if (cudaMemsetAsync(ws, 0, rl.zero_bytes, st) != cudaSuccess) {
        rc = AAREN_ERR_CUDA;
    } else {
        char *base = static_cast<char *>(ws);
        ReduceParams p;
        p.q = q; p.K = K; p.V = V; p.o_last = o_last;
        p.m_in = m_in; p.u_in = u_in; p.w_in = w_in;
        p.m_out = m_out; p.u_out = u_out; p.w_out = w_out;
        p.counts = reinterpret_cast<unsigned *>(base);
        p.parts = reinterpret_cast<float *>(base + rl.parts_off);
        p.N = N;
        p.heads = BH;
        p.P = 1;
        p.seg = kReduceRows;
        p.part_slots = BH * rl.P_max;
        p.status = nullptr;
#ifdef AAREN_CHECKED
        if (cudaGetSymbolAddress(reinterpret_cast<void **>(&p.status), g_status) != cudaSuccess) {
            if (owned) cudaFreeAsync(ws, st);
            return AAREN_ERR_CUDA;
        }
#endif
        rc = dispatch_reduce(p, rl.P_max, d, dtype, st);
    }
    if (owned && cudaFreeAsync(ws, st) != cudaSuccess && rc == AAREN_OK) rc = AAREN_ERR_CUDA;
    return rc;
}

aaren_status_t aaren_scan_forward_ex(const void *q, const void *K, const void *V, void *O,
                                     int64_t B, int64_t H, int64_t N, int64_t d, int32_t dtype,
                                     const float *m_in, const float *u_in, const float *w_in,
                                     float *m_out, float *u_out, float *w_out, void *workspace,
                                     size_t workspace_bytes, void *stream)
{
    return scan_forward_impl(q, K, V, O, B, H, N, d, dtype, m_in, u_in, w_in, m_out, u_out, w_out,
                             nullptr, workspace, workspace_bytes, stream);
}

aaren_status_t aaren_scan_forward_stats(const void *q, const void *K, const void *V, void *O,
                                        float *stats, int64_t B, int64_t H, int64_t N, int64_t d,
                                        int32_t dtype, void *workspace, size_t workspace_bytes,
                                        void *stream)
{
    if (N > 0 && stats == nullptr) return AAREN_ERR_INVALID;
    if (!aligned(stats, 8)) return AAREN_ERR_INVALID;
    return scan_forward_impl(q, K, V, O, B, H, N, d, dtype, nullptr, nullptr, nullptr, nullptr,
                             nullptr, nullptr, stats, workspace, workspace_bytes, stream);
}

aaren_status_t aaren_scan_forward(const void *q, const void *K, const void *V, void *O, int64_t B,
                                  int64_t H, int64_t N, int64_t d, int32_t dtype, void *stream)
{
    return aaren_scan_forward_ex(q, K, V, O, B, H, N, d, dtype, nullptr, nullptr, nullptr, nullptr,
                                 nullptr, nullptr, nullptr, 0, stream);
}

aaren_status_t aaren_state_init(float *m, float *u, float *w, int64_t n, int64_t d, void *stream)
{
    if (!supported_d(d)) return AAREN_ERR_UNSUPPORTED;
    if (n < 0) return AAREN_ERR_INVALID;
    int64_t nd;
    if (!mul_ok(n, d, &nd)) return AAREN_ERR_INVALID;
    if (n == 0) return AAREN_OK;
    if (m == nullptr || u == nullptr || w == nullptr) return AAREN_ERR_INVALID;
    if (check_state(m, u, w) != AAREN_OK) return AAREN_ERR_INVALID;
    return launch_state_init(m, u, w, n, d, static_cast<cudaStream_t>(stream));
}

aaren_status_t aaren_step(const void *q, float *m, float *u, float *w, const void *k_t,
                          const void *v_t, void *o_t, int64_t n, int64_t d, int32_t dtype,
                          void *stream)
{
    if (!supported_dtype(dtype) || !supported_d(d)) return AAREN_ERR_UNSUPPORTED;
    if (n < 0) return AAREN_ERR_INVALID;
    int64_t nd, threads;
    if (!mul_ok(n, d, &nd) || !mul_ok(n, 32, &threads) || threads / 256 >= INT_MAX) return AAREN_ERR_INVALID;
    if (n == 0) return AAREN_OK;
    if (q == nullptr || k_t == nullptr || v_t == nullptr || o_t == nullptr || m == nullptr ||
        u == nullptr || w == nullptr)
        return AAREN_ERR_INVALID;
    if (!aligned(q, 16) || !aligned(k_t, 16) || !aligned(v_t, 16) || !aligned(o_t, 16))
        return AAREN_ERR_INVALID;
    if (check_state(m, u, w) != AAREN_OK) return AAREN_ERR_INVALID;
    unsigned *status = nullptr;   // the step's only device-side report is a bounds violation
#ifdef AAREN_CHECKED
    if (cudaGetSymbolAddress(reinterpret_cast<void **>(&status), g_status) != cudaSuccess) return AAREN_ERR_CUDA;
#endif
    StepParams p;
    p.q = q; p.m = m; p.u = u; p.w = w; p.k = k_t; p.v = v_t; p.o = o_t; p.n = n;
    p.status = status;
    p.probe = g_bounds_probe.load();
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (d) {
    case 16: return dispatch_step_dtype<16>(p, dtype, st);
    case 32: return dispatch_step_dtype<32>(p, dtype, st);
    case 64: return dispatch_step_dtype<64>(p, dtype, st);
    case 128: return dispatch_step_dtype<128>(p, dtype, st);
    default: return AAREN_ERR_UNSUPPORTED;
    }
}

aaren_status_t aaren_check(void *stream)
{
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return AAREN_ERR_CUDA;
    unsigned bits = 0;
    if (cudaMemcpyFromSymbol(&bits, g_status, sizeof(bits)) != cudaSuccess) return AAREN_ERR_CUDA;
    if (bits == 0) return AAREN_OK;
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_status, &zero, sizeof(zero)) != cudaSuccess) return AAREN_ERR_CUDA;
    if (bits & STATUS_BOUNDS) return AAREN_ERR_BOUNDS;
    if (bits & STATUS_LOAD_TIMEOUT) return AAREN_ERR_LOAD_TIMEOUT;
    return AAREN_ERR_LOOKBACK_TIMEOUT;
}

const char *aaren_status_string(int32_t status)
{
    switch (status) {
    case AAREN_OK: return "ok";
    case AAREN_ERR_INVALID: return "invalid argument";
    case AAREN_ERR_UNSUPPORTED: return "unsupported d or dtype";
    case AAREN_ERR_CUDA: return "CUDA runtime error";
    case AAREN_ERR_LOOKBACK_TIMEOUT: return "device: cross-block carry wait gave up";
    case AAREN_ERR_BOUNDS: return "device (checked build): an index outside its buffer, access skipped";
    case AAREN_ERR_LOAD_TIMEOUT: return "device: bulk copy or in-block hand-off did not complete";
    case AAREN_ERR_WORKSPACE: return "workspace too small or misaligned";
    default: return "unknown status";
    }
}

int32_t aaren_abi_version(void) { return 2; }

aaren_status_t aaren_debug_set_fault(int64_t never_publish_chunk, int64_t wait_limit_ns)
{
    g_fault_chunk.store(never_publish_chunk < 0 ? -1 : never_publish_chunk);
    g_wait_limit_ns.store(wait_limit_ns <= 0 ? kDefaultWaitLimitNs : wait_limit_ns);
    return AAREN_OK;
}

aaren_status_t aaren_debug_drop_arrival(int64_t chunk)
{
    g_drop_chunk.store(chunk < 0 ? -1 : chunk);
    return AAREN_OK;
}

aaren_status_t aaren_debug_bounds_probe(int64_t offset)
{
    g_bounds_probe.store(offset);
    return AAREN_OK;
}

int32_t aaren_checked_build(void)
{
#ifdef AAREN_CHECKED
    return 1;
#else
    return 0;
#endif
}

int64_t aaren_scan_chunk_tokens(int64_t d, int32_t dtype)
{
    if (!supported_d(d) || !supported_dtype(dtype)) return 0;
    return chunk_tokens(d, dtype);
}

int64_t aaren_backward_chunk_tokens(int64_t d, int32_t dtype)
{
    if (!supported_d(d) || !supported_dtype(dtype)) return 0;
    return bwd_chunk_tokens(d, dtype);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free scan: the same scan with its cross-block carry workspace in
// a fixed device array of this library instead of memory the caller or the
// stream-ordered allocator provides.
// ---------------------------------------------------------------------------

static __device__ __align__(256) unsigned char g_noalloc_scratch[AAREN_NOALLOC_SCRATCH_BYTES];

namespace aaren {
namespace {

constexpr int kMaxNoallocDevices = 64;
std::atomic<void *> g_noalloc_scratch_ptr[kMaxNoallocDevices];

// Device address of g_noalloc_scratch on the current device, looked up once
// per device (the array's name in host code is only a host-side handle).
aaren_status_t noalloc_scratch(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxNoallocDevices)
        return AAREN_ERR_CUDA;
    void *ptr = g_noalloc_scratch_ptr[dev].load();
    if (ptr == nullptr) {
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
            return AAREN_ERR_CUDA;
        g_noalloc_scratch_ptr[dev].store(ptr);
    }
    *out = ptr;
    return AAREN_OK;
}

}  // namespace
}  // namespace aaren

extern "C" aaren_status_t aaren_scan_forward_noalloc(const void *q, const void *K, const void *V,
                                                     void *O, int64_t B, int64_t H, int64_t N,
                                                     int64_t d, int32_t dtype, void *stream)
{
    // Sizes first: a problem whose workspace exceeds the array is rejected
    // before any pointer is looked at or any CUDA call is made.
    if (!supported_dtype(dtype) || !supported_d(d)) return AAREN_ERR_UNSUPPORTED;
    if (B < 0 || H < 0 || N < 0) return AAREN_ERR_INVALID;
    const size_t need = aaren_scan_workspace_bytes(B, H, N, d);
    if (need == SIZE_MAX) return AAREN_ERR_INVALID;   // the shape overflows
    if (need > AAREN_NOALLOC_SCRATCH_BYTES) return AAREN_ERR_WORKSPACE;
    void *scratch = nullptr;
    const aaren_status_t rc = noalloc_scratch(&scratch);
    if (rc != AAREN_OK) return rc;
    // The regular path with a caller workspace allocates nothing: it checks
    // the pointers, zeroes the ticket and flags of the workspace (a small
    // kernel) and launches.
    return aaren_scan_forward_ex(q, K, V, O, B, H, N, d, dtype, nullptr, nullptr, nullptr, nullptr,
                                 nullptr, nullptr, scratch, AAREN_NOALLOC_SCRATCH_BYTES, stream);
}
