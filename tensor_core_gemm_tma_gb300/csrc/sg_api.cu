// sg_api.cu -- host side of the C ABI declared in include/stage_gemm.h:
// argument checks, the launch plan (tile width, stage count, persistent grid),
// the TMA tensor-map builder, the kernel launch, and the host-buffer entry
// (chunked copies overlapped with the GEMMs).
//
// Every argument check runs before the first CUDA call, so a rejected call
// never touches the device.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "sg_launch.cuh"
#include "stage_gemm.h"

namespace {

constexpr int kMaxDevices = 64;
// Cluster row blocks swept together by the tile raster (L2 reuse of the B
// tiles they share).  12 measured best on GB300 among 4-24 (8192^3 bf16 and
// FP8, 4096^3, 16384 x 8192 x 4096, 6144 x 12288 x 4096): 0-4% over 8.
// STAGE_GEMM_GROUP_M overrides it at load (tuning only: the order of tiles
// never changes a result).
const int kGroupM = [] {
    const char* e = std::getenv("STAGE_GEMM_GROUP_M");
    const int x = e ? std::atoi(e) : 0;
    return (x >= 1 && x <= 64) ? x : 12;
}();

struct DevState {
    bool ready = false;
    int sm_count = 0;
    int smem_optin = 0;   // max dynamic shared memory per block
    int smem_per_sm = 0;
    int major = 0, minor = 0;
    int* status = nullptr;  // device status word (4 bytes, library-owned)
    // per kernel instantiation [tile width][output type][mode - 1][residual]:
    bool attr_done[2][3][3][6][2] = {};    // [8-bit][tile width][output type][mode - 1][residual]: attribute set
    int max_clusters[2][3][3][6][2] = {};  // the same index: co-resident clusters (0: not queried)
    // sg_gemm_host: library-owned copy streams, a second compute stream and
    // events, created on first use
    cudaStream_t h2d = nullptr, d2h = nullptr, comp = nullptr;
    // the library's stream-ordered memory pool (scratch_pool), created on first use
    int dev = 0;
    bool pool_tried = false;
    cudaMemPool_t pool = nullptr;
    cudaEvent_t ev_fork = nullptr, ev_in = nullptr, ev_gemm = nullptr, ev_out = nullptr, ev_comp = nullptr;
};

std::mutex g_mu;
std::mutex g_host_mu;  // serialises sg_gemm_host calls while they queue work
DevState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

uint64_t initial_wait_limit() {
    const char* e = std::getenv("STAGE_GEMM_WAIT_LIMIT_MS");
    if (e && *e) {
        char* end = nullptr;
        const double ms = std::strtod(e, &end);
        if (end != e && ms > 0) return static_cast<uint64_t>(ms * 1e6);
    }
    return 2000000000ull;  // 2 s
}
std::atomic<uint64_t> g_wait_limit_ns{initial_wait_limit()};

// Test hook (not in the public header): the next launches skip copying the
// K chunk with this global index, so the MMA's wait for it runs out.
std::atomic<int64_t> g_skip_load{-1};

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
int elem_bytes(int dt) { return dt == SG_F32 ? 4 : dt == SG_E4M3 ? 1 : 2; }
bool valid_in(int dt) { return dt == SG_F16 || dt == SG_BF16 || dt == SG_E4M3; }
bool valid_out(int dt) { return dt == SG_F32 || dt == SG_F16 || dt == SG_BF16; }
bool valid_epi(int e) { return e == SG_EPI_NONE || e == SG_EPI_RELU || e == SG_EPI_BIAS_RELU; }

// [p, p + n) and [q, q + m) overlap (empty ranges never do)
bool overlap(const void* p, uint64_t n, const void* q, uint64_t m) {
    if (!p || !q || n == 0 || m == 0) return false;
    const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(q);
    return a < b + m && b < a + n;
}

uint64_t span_bytes(int64_t rows, int64_t cols, int64_t ld, int esize) {
    if (rows <= 0 || cols <= 0) return 0;
    return static_cast<uint64_t>((rows - 1) * ld + cols) * static_cast<uint64_t>(esize);
}

// Host-only argument checks (no CUDA calls).
int check_args(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb, const void* C,
               int64_t ldc, int in_dtype, int out_dtype, int epilogue, const float* bias, int stages) {
    if (!valid_in(in_dtype) || !valid_out(out_dtype) || !valid_epi(epilogue)) return SG_ERR_DTYPE;
    if (M < 0 || N < 0 || K < 0) return SG_ERR_ARG;
    const int64_t lim = 0x7FFFFFFF;
    if (M > lim || N > lim || K > lim || lda > lim || ldb > lim || ldc > lim) return SG_ERR_ARG;
    if (stages < 0 || stages > SG_MAX_STAGES) return SG_ERR_STAGES;
    if ((epilogue == SG_EPI_BIAS_RELU) != (bias != nullptr)) return SG_ERR_ARG;
    if (M == 0 || N == 0) return SG_OK;
    if (!C || ldc < N) return SG_ERR_ARG;
    if (K > 0 && (!A || !B || lda < K || ldb < N)) return SG_ERR_ARG;
    if (cdiv(M, sg::BM) * cdiv(N, 64) > lim) return SG_ERR_ARG;
    const uint64_t c_span = span_bytes(M, N, ldc, elem_bytes(out_dtype));
    if (K > 0) {
        const int ies = elem_bytes(in_dtype);
        if (overlap(C, c_span, A, span_bytes(M, K, lda, ies)) || overlap(C, c_span, B, span_bytes(K, N, ldb, ies)))
            return SG_ERR_ALIAS;
    }
    if (bias && overlap(C, c_span, bias, static_cast<uint64_t>(N) * 4)) return SG_ERR_ALIAS;
    // Every pointer must sit on a boundary of its own elements (2 bytes for
    // 16-bit operands, the output type's size for C, 4 for the fp32 bias):
    // the element loads and masked element stores that take over where TMA
    // cannot address an operand or C access single elements, and a
    // misaligned element access faults on the GPU.  Anything coarser is
    // handled (TMA when legal, element accesses otherwise).
    const uintptr_t emask = static_cast<uintptr_t>(elem_bytes(in_dtype) - 1);
    if (K > 0 && ((reinterpret_cast<uintptr_t>(A) & emask) || (reinterpret_cast<uintptr_t>(B) & emask)))
        return SG_ERR_ALIGN;
    if (reinterpret_cast<uintptr_t>(C) & static_cast<uintptr_t>(elem_bytes(out_dtype) - 1)) return SG_ERR_ALIGN;
    if (bias && (reinterpret_cast<uintptr_t>(bias) & 3u)) return SG_ERR_ALIGN;
    return SG_OK;
}

// The residual's host-only checks (sg_gemm_residual, sg_gemm_ex, sg_gemm_host).
int check_residual(int64_t M, int64_t N, const void* R, int64_t ldr, const void* C, int64_t ldc, int out_dtype) {
    if (!R || ldr < N || ldr > 0x7FFFFFFF) return SG_ERR_ARG;
    const int oes = elem_bytes(out_dtype);
    if (reinterpret_cast<uintptr_t>(R) % oes) return SG_ERR_ALIGN;
    // R may be C itself (each element is read before it is written); any
    // other overlap of the two would race
    const bool same = (R == C && ldr == ldc);
    if (!same && overlap(C, span_bytes(M, N, ldc, oes), R, span_bytes(M, N, ldr, oes))) return SG_ERR_ALIAS;
    return SG_OK;
}

// An operand can be copied by TMA when its base is 16-byte aligned and its
// row pitch is a multiple of 16 bytes (a single row has no pitch).
bool tma_legal(const void* X, int64_t rows, int64_t ld, int esz) {
    return (reinterpret_cast<uintptr_t>(X) & 15) == 0 && (rows <= 1 || (ld * esz) % 16 == 0);
}

int ensure_encode_fn() {
    if (g_encode) return SG_OK;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
        return SG_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return SG_OK;
}

// Per-device set-up, once: properties, the status word, the encoder.
int device_state(DevState** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SG_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    DevState& st = g_dev[dev];
    if (!st.ready) {
        if (cudaDeviceGetAttribute(&st.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&st.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return SG_ERR_CUDA;
        if (st.major != 10 || st.minor != 3) return SG_ERR_ARCH;
        if (cudaDeviceGetAttribute(&st.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&st.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&st.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) !=
                cudaSuccess)
            return SG_ERR_CUDA;
        if (int rc = ensure_encode_fn(); rc != SG_OK) return rc;
        if (cudaMalloc(&st.status, sizeof(int)) != cudaSuccess) return SG_ERR_CUDA;
        if (cudaMemset(st.status, 0, sizeof(int)) != cudaSuccess) return SG_ERR_CUDA;
        st.dev = dev;
        st.ready = true;
    }
    *out = &st;
    return SG_OK;
}

// The library's stream-ordered memory pool on this device, created on first
// use.  sg_gemm_host's staging buffer and the 16-byte-pitch copies of
// operands come from it.  Blocks freed on a stream stay in the pool (no
// release threshold), so a later call of the same size maps no new memory;
// the device's default pool, whose threshold is 0, would return them at
// every synchronisation and map them again on the next call.  The pool and
// what it holds last until the process exits.
cudaMemPool_t scratch_pool(DevState& st) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!st.pool_tried) {
        st.pool_tried = true;
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = st.dev;
        cudaMemPool_t pool = nullptr;
        if (cudaMemPoolCreate(&pool, &props) == cudaSuccess) {
            uint64_t keep = UINT64_MAX;
            if (cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep) == cudaSuccess) {
                st.pool = pool;
            } else {
                cudaMemPoolDestroy(pool);
            }
        }
        cudaGetLastError();  // a device without pools: the default pool serves
    }
    return st.pool;
}

// A stream-ordered allocation from the library's pool; from the device's
// default pool while `s` is being captured into a graph (the allocation then
// becomes the graph's own) or where the library has no pool.  Freed with
// cudaFreeAsync either way.
cudaError_t pool_alloc(DevState& st, void** p, size_t bytes, cudaStream_t s) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) return cudaErrorUnknown;
    cudaMemPool_t pool = cap == cudaStreamCaptureStatusNone ? scratch_pool(st) : nullptr;
    return pool ? cudaMallocFromPoolAsync(p, bytes, pool, s) : cudaMallocAsync(p, bytes, s);
}

// The copy streams and events of sg_gemm_host, once per device.
int host_streams(DevState& st) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (st.h2d) return SG_OK;
    cudaStream_t q[3] = {};
    cudaEvent_t e[5] = {};
    bool ok = true;
    for (auto& x : q) ok = ok && cudaStreamCreateWithFlags(&x, cudaStreamNonBlocking) == cudaSuccess;
    for (auto& ev : e) ok = ok && cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        for (auto& x : q)
            if (x) cudaStreamDestroy(x);
        for (auto& ev : e)
            if (ev) cudaEventDestroy(ev);
        return SG_ERR_CUDA;
    }
    st.ev_fork = e[0];
    st.ev_in = e[1];
    st.ev_gemm = e[2];
    st.ev_out = e[3];
    st.ev_comp = e[4];
    st.d2h = q[1];
    st.comp = q[2];
    st.h2d = q[0];  // last: a non-null h2d marks the set as complete
    return SG_OK;
}

// Row chunks of sg_gemm_host: about one per 32 MB of copies, at most 16,
// each a whole number of 256-row pair tiles; STAGE_GEMM_HOST_CHUNKS (1..64)
// overrides the count.  On GB300 (host link ~210 GB/s each way) 8-24 chunks
// were within 2% of each other for 8192^3 and for M=518400, K=96, N=384.
int64_t host_chunk_rows(int64_t M, uint64_t copy_bytes) {
    int64_t n = static_cast<int64_t>(copy_bytes / (32ull << 20));
    n = std::max<int64_t>(1, std::min<int64_t>(16, n));
    if (const char* e = std::getenv("STAGE_GEMM_HOST_CHUNKS")) {
        const int x = std::atoi(e);
        if (x >= 1 && x <= 64) n = x;
    }
    const int64_t rows = cdiv(cdiv(M, n), 2 * sg::BM) * (2 * sg::BM);
    return std::max<int64_t>(rows, 1);
}

// A launch configuration chosen by sg_tune or given to sg_gemm_ex: every
// non-zero field overrides the planner's heuristic.  tail_split < 0 never
// splits the last wave.  A strict choice (sg_gemm_ex) must be honoured as
// given: a tile width or mode the problem cannot take is SG_ERR_CONFIG
// instead of the planner's fallback.
struct Choice {
    int bn = 0, mode = 0, stages = 0, group_m = 0, tail_split = 0;
    bool strict = false;
};

// Tuning cache: the fastest configuration measured for each problem key.
using TuneKey = std::tuple<int, int64_t, int64_t, int64_t, int, int, int, int, int, int>;
std::map<TuneKey, Choice> g_tuned;

TuneKey tune_key(int dev, int64_t M, int64_t N, int64_t K, int in_dtype, int out_dtype, int epi, bool a_tma,
                 bool b_tma, bool c_tma) {
    return TuneKey(dev, M, N, K, in_dtype, out_dtype, epi, a_tma, b_tma, c_tma);
}

struct Plan {
    int bn = 128;      // accumulator width (the MMA's N)
    int tw = 128;      // tile width: bn, or 2 * bn for mode 6's two accumulators
    int block_k = 64;  // K elements per stage (128 bytes of K)
    int group_m = 12;
    int mode = 1;  // 1: single CTA, 3: paired MMA, 4: resident B, 5: decoded panel, 6: wide paired tiles
    int cm = 1;    // CTAs per cluster along M
    int stages = 0, max_stages = 0;
    int ring_group = 1;  // ring slots sharing one full and one empty barrier
    int64_t units = 0, full_units = 0;  // work units launched; those of whole tiles (the rest: half tiles)
    int64_t m_blocks = 0, n_blocks = 0, tiles = 0, k_chunks = 0;
    int grid = 0;
    int smem = 0;
    int tmem_cols = 0;
    int tma_store = 0;
    int a_tma = 1, b_tma = 1;  // operand copied by TMA (1) or by element loads (0)
};

// Modes 4 and 5's shared memory: the resident B (k_chunks x n_blocks blocks
// of bn columns by 128 bytes of K), a ring of A tiles (k_chunks chunks
// each), the staging buffers, mode 5's per-column scales and biases (fp32,
// n_blocks * bn of each) or mode 4's biases (with a bias), and the barriers.
int64_t smem_panel(int bn, int stages, int64_t k_chunks, int64_t n_blocks, bool decode = false, bool bias = false) {
    return k_chunks * n_blocks * bn * sg::BK_BYTES + stages * k_chunks * sg::A_STAGE_BYTES +
           sg::EPI_WARPS * sg::EPI_BUF_BYTES + (decode ? n_blocks * bn * 8 : bias ? n_blocks * bn * 4 : 0) +
           sg::BAR_AREA + sg::SMEM_ALIGN;
}

int smem_for(int bn, int stages, int mode) {
    if (mode == 6) {  // each CTA stages half of each of the tile's two accumulators' B
        return bn == 256 ? sg::Layout<256, 256>::smem_bytes(stages) : -1;
    }
    if (mode == 3) {  // each CTA stages half of B
        switch (bn) {
            case 128: return sg::Layout<128, 64>::smem_bytes(stages);
            case 256: return sg::Layout<256, 128>::smem_bytes(stages);
            default: return -1;
        }
    }
    switch (bn) {
        case 128: return sg::Layout<128>::smem_bytes(stages);
        case 192: return sg::Layout<192>::smem_bytes(stages);
        case 256: return sg::Layout<256>::smem_bytes(stages);
        default: return -1;
    }
}

// Tile width forced by sg_test_set_tile_n or, at load, the environment
// variable STAGE_GEMM_TILE_N (128, 192 or 256; 0: the planner's choice).  A
// tuning knob only: every width sums the same products for each output
// element in the same K order.
int valid_bn(int x) { return (x == 128 || x == 192 || x == 256) ? x : 0; }
std::atomic<int> g_force_bn{[] {
    const char* e = std::getenv("STAGE_GEMM_TILE_N");
    return e ? valid_bn(std::atoi(e)) : 0;
}()};
int forced_bn() { return g_force_bn.load(); }

// Splitting a short last wave of 256-column tiles into half tiles, set by
// sg_test_set_tail_split or, at load, the environment variable
// STAGE_GEMM_TAIL_SPLIT (0: never; 1: where it pays, the default).
std::atomic<int> g_tail_split{[] {
    const char* e = std::getenv("STAGE_GEMM_TAIL_SPLIT");
    return (e && std::atoi(e) == 0) ? 0 : 1;
}()};

// Whether operands without a TMA-legal layout may be copied to 16-byte
// pitches before the launch (sg_test_set_repack; 1 by default).
std::atomic<int> g_repack{1};

// Kernel mode forced by sg_test_set_cluster or, at load, the environment
// variable STAGE_GEMM_CLUSTER (1: single CTA, 3: paired MMA, 4: resident B,
// 6: wide paired tiles; 0: the planner's choice).
bool valid_mode(int x) { return x == 1 || x == 3 || x == 4 || x == 6; }
// Tile widths an sg_config may ask for (512: mode 6's two 256-column accumulators).
bool valid_tile(int x) { return valid_bn(x) || x == 512; }
std::atomic<int> g_force_mode{[] {
    const char* e = std::getenv("STAGE_GEMM_CLUSTER");
    const int x = e ? std::atoi(e) : 0;
    return valid_mode(x) ? x : 0;
}()};

// Waves of `units` work units over `slots` clusters, the last wave counted
// half when it would be split into half-width units (fills at most half of
// the slots; see the tail split below).
double wave_count(int64_t units, int64_t slots, bool splittable) {
    const int64_t full = units / slots, tail = units % slots;
    double w = static_cast<double>(full);
    if (tail) w += (splittable && full > 0 && 2 * tail <= slots) ? 0.5 : 1.0;
    return w;
}

int make_plan(const DevState& st, int64_t M, int64_t N, int64_t K, int in_dtype, int out_dtype, const void* C,
              int64_t ldc, int stages, bool a_tma, bool b_tma, Plan* pl, const Choice* choice = nullptr,
              bool decode = false, bool residual = false, bool bias = false) {
    const int esz = elem_bytes(in_dtype);
    const int boxc = 128 / esz;  // B columns per 128-byte box: tile widths and CTA shares are multiples
    pl->a_tma = a_tma ? 1 : 0;
    pl->b_tma = b_tma ? 1 : 0;
    pl->m_blocks = cdiv(M, sg::BM);
    pl->block_k = sg::BK_BYTES / esz;
    pl->k_chunks = cdiv(K, pl->block_k);
    // Tile width: the one of 256 / 192 / 128 with the least estimated time,
    // counted as whole waves of tiles over the SMs times the time of one tile
    // (its width over its throughput relative to 256 columns).  Narrower tiles
    // stage more operand bytes per product, and with every SM loading that
    // costs throughput: on GB300 (8192^3, 8192^2 x 2048, 4096^3) 192 columns
    // (single CTAs, a 4-slot ring) ran at ~0.64 of 256 and 128 (CTA pairs,
    // 8 slots) at ~0.65.  Those ratios are rough, so a narrower width must
    // win by 5%.  A
    // short K loop (<= 4 chunks) makes the epilogue the bottleneck: keep 128,
    // whose four tensor-memory accumulators overlap it best.
    int bn = 128;
    if (pl->k_chunks > 4) {
        double best = 0.0;
        for (int cand : {256, 192, 128}) {
            if (cand % boxc) continue;
            const double rel = cand == 256 ? 1.0 : cand == 192 ? 0.64 : 0.65;
            const int64_t waves = cdiv(pl->m_blocks * cdiv(N, cand), static_cast<int64_t>(st.sm_count));
            const double cost = static_cast<double>(waves) * cand / rel;
            if (best == 0.0 || cost < 0.95 * best) {
                best = cost;
                bn = cand;
            }
        }
    }
    if (forced_bn()) bn = forced_bn();
    // a 512-column tile is mode 6: two 256-column accumulators
    bool wide = false;
    if (choice && choice->bn) {
        wide = choice->bn == 512;
        bn = wide ? 256 : choice->bn;
    }
    if (choice && choice->mode == 6) {
        wide = true;
        if (!choice->bn) bn = 256;
    }
    const bool bn_forced = forced_bn() || (choice && (choice->bn || choice->mode == 6));
    if (bn % boxc) return SG_ERR_CONFIG;  // a forced width that is not whole 128-byte B boxes
    pl->bn = bn;
    pl->group_m = (choice && choice->group_m) ? choice->group_m : kGroupM;
    const bool pairable = (bn / boxc) % 2 == 0;  // each CTA of a pair owns whole boxes of B
    // Pairs of CTAs compute 256-row tiles with the paired MMA when the K loop
    // is long enough for operand traffic to matter: each SM then stages only
    // its half of B.  A pair tile is two SMs' work, so pairing keeps as many
    // SMs busy as single-CTA tiles do.
    int mode = (pl->k_chunks >= 8 && pl->m_blocks >= 2 && pairable) ? 3 : 1;
    // Mode 6 (a CTA pair computes 256 x 512 as two 256-column accumulators:
    // a quarter fewer operand bytes per product and half as many tiles)
    // instead of paired 256-column tiles when its waves cost less, counting
    // its per-SM throughput at full load as 1.08 of theirs (measured on
    // GB300: 8192^3 bf16 +7.9%, FP8 +3.9%, 16384 x 8192 x 4096 +3.3%,
    // 6144 x 12288 x 4096 +1.4%, 8192^2 x 2048 +1.3%; 4096^3 -2 to 0% and
    // 2048^3 -29%, left out by requiring three full waves of wide tiles).
    // Only with a long K loop (the tile boundary, where the second
    // accumulator waits for the previous tile's epilogue to read it, then
    // weighs little), a 16-bit output and no residual (there the epilogue
    // hands the accumulator back before storing).
    bool auto_wide = false;
    if (mode == 3 && bn == 256 && !bn_forced && pl->k_chunks >= 32 && out_dtype != SG_F32 && !residual && a_tma &&
        b_tma && !decode) {
        const int64_t clusters = st.sm_count / 2, mc = cdiv(pl->m_blocks, 2);
        const int64_t wide_tiles = mc * cdiv(N, 512);
        const double c3 = wave_count(mc * cdiv(N, 256), clusters, esz == 2) * 256.0;
        const double c6 = wave_count(wide_tiles, clusters, true) * 512.0 / 1.08;
        // at least three full waves of wide tiles: with fewer (4096^3: 1.7)
        // the estimate of the last wave was off by more than the margin
        auto_wide = wide_tiles >= 3 * clusters && c6 < 0.98 * c3;
    }
    // Mode 4 (resident B) when B is small: at most 2 K chunks and 4 column
    // blocks of 128, so all of B fits next to a ring of at least 2 A tiles,
    // and there are enough row tiles to keep every SM busy.
    const int64_t nb128 = cdiv(N, 128);
    const bool panel_ok = a_tma && b_tma && pl->k_chunks <= 2 && nb128 <= 4 &&
                          smem_panel(128, 2, pl->k_chunks, nb128, false, bias) <= st.smem_optin;
    if (panel_ok && pl->m_blocks >= st.sm_count && !bn_forced) mode = 4;
    auto legal = [&](int m) {
        return m == 1 || (m == 3 && pairable) || (m == 4 && panel_ok) || (m == 6 && bn == 256 && a_tma && b_tma);
    };
    if (auto_wide && legal(6)) mode = 6;
    if (const int f = g_force_mode.load(); f && legal(f)) mode = f;
    if (choice && choice->mode && legal(choice->mode)) mode = choice->mode;
    if (wide && legal(6)) mode = 6;
    if (!a_tma || !b_tma) mode = 1;  // element-load staging runs in single-CTA mode
    if (decode) {
        // mode 5: the integer-coded B is decoded into mode 4's resident panel,
        // so B must fit there (it is never read by TMA)
        if (!(a_tma && pl->k_chunks <= 2 && nb128 <= 4 &&
              smem_panel(128, 1, pl->k_chunks, nb128, true) <= st.smem_optin))
            return SG_ERR_ARG;
        mode = 5;
    }
    const bool panel = mode == 4 || mode == 5;
    if (panel) {
        bn = 128;
        pl->bn = bn;
        pl->n_blocks = nb128;
    }
    pl->mode = mode;
    pl->tw = mode == 6 ? 2 * bn : bn;
    if (!panel) pl->n_blocks = cdiv(N, pl->tw);
    pl->cm = (mode == 3 || mode == 6) ? 2 : 1;
    const int cm = pl->cm;
    // work units handed out by the persistent loop: cluster tiles (modes 1, 3, 6)
    // or row tiles covering every column block (modes 4, 5)
    pl->tiles = panel ? pl->m_blocks : cdiv(pl->m_blocks, cm) * pl->n_blocks;
    int maxs = 0;
    for (int s = 1; s <= SG_MAX_STAGES; ++s) {
        const int64_t need =
            panel ? smem_panel(bn, s, pl->k_chunks, pl->n_blocks, mode == 5, bias) : smem_for(bn, s, mode);
        if (need <= st.smem_optin) maxs = s;
    }
    pl->max_stages = maxs;
    if (maxs == 0) return SG_ERR_STAGES;
    if (stages == 0 && choice && choice->stages) stages = std::min(choice->stages, maxs);
    if (stages == 0) stages = maxs;
    if (stages > maxs) return SG_ERR_STAGES;
    pl->stages = stages;
    // The MMA warp's wait on a ring barrier stalls its issue long enough for
    // the tensor pipe to drain: pairing slots on one barrier halves those
    // waits (5-6% on 8192^3 and FP8 8192^3, ~6% on 4096^3 on GB300).  A pair
    // is refilled only when both of its slots are free, so the ring keeps at
    // least three pairs (three chunks in flight: two pairs measured slower
    // than single slots).  Both operands must arrive by TMA, whose bytes the
    // barrier counts; the grouping never changes which MMAs run or their
    // order, so C keeps its bits.
    pl->ring_group = (!panel && a_tma && b_tma && stages >= 6 && stages % 2 == 0) ? 2 : 1;
    pl->smem = panel ? static_cast<int>(smem_panel(bn, stages, pl->k_chunks, pl->n_blocks, mode == 5, bias))
                     : smem_for(bn, stages, mode);
    pl->tmem_cols = sg::TMEM_COLS;
    // Two CTAs on one SM would each hold half the tensor memory or wait for
    // it; keep one persistent CTA per SM by asking for more than half of the
    // SM's shared memory.
    if (pl->tmem_cols > 256 && pl->smem <= st.smem_per_sm / 2) pl->smem = st.smem_per_sm / 2 + 1024;
    const int64_t clusters = st.sm_count / cm;
    // A last wave that fills at most half of the clusters takes as long as a
    // full one.  Its tiles, when 256 columns wide (16-bit operands, both by
    // TMA), are split into two 128-column units each, so that wave spreads
    // over twice as many clusters and takes about half as long (the other
    // waves are unchanged).  Each output element is still computed by one
    // unit, summing the same products in the same K order: C keeps its bits.
    pl->units = pl->full_units = pl->tiles;
    const int64_t tail = pl->tiles % clusters;
    const bool split_ok = g_tail_split.load() && !(choice && choice->tail_split < 0);
    const bool splittable = mode == 6 || (esz == 2 && bn == 256);  // halves of whole B boxes per CTA
    if (split_ok && !panel && splittable && a_tma && b_tma && pl->k_chunks > 0 &&
        pl->tiles > clusters && tail > 0 && 2 * tail <= clusters) {
        pl->full_units = pl->tiles - tail;
        pl->units = pl->full_units + 2 * tail;
    }
    pl->grid = static_cast<int>((pl->units < clusters ? pl->units : clusters) * cm);
    const int oes = elem_bytes(out_dtype);
    pl->tma_store = ((reinterpret_cast<uintptr_t>(C) & 15) == 0 && (M == 1 || (ldc * oes) % 16 == 0)) ? 1 : 0;
    return SG_OK;
}

CUtensorMapDataType tmap_dtype(int dt) {
    switch (dt) {
        case SG_E4M3: return CU_TENSOR_MAP_DATA_TYPE_UINT8;  // bytes are moved, never interpreted
        case SG_F16: return CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
        case SG_BF16: return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        default: return CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    }
}

// 2-D row-major tensor [outer][inner] with a pitch of `pitch_bytes`, copied in
// boxes of box_inner x box_outer elements with the 128-byte swizzle.
int encode_2d(CUtensorMap* tm, int dt, const void* ptr, int64_t inner, int64_t outer, int64_t pitch_bytes,
              uint32_t box_inner, uint32_t box_outer) {
    if (outer == 1) pitch_bytes = (inner * elem_bytes(dt) + 15) / 16 * 16;  // unused, but must be legal
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(pitch_bytes)};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = g_encode(tm, tmap_dtype(dt), 2, const_cast<void*>(ptr), dims, strides, box, estr,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? SG_OK : SG_ERR_CUDA;
}

// Launch the instantiation the plan names (it lives in one of the
// sg_inst_*.cu units).
int launch_plan(DevState& st, int out_dtype, const Plan& pl, const CUtensorMap& ta, const CUtensorMap& tb,
                const CUtensorMap& tc, const CUtensorMap& tr, const sg::Params& prm, bool residual,
                cudaStream_t stream) {
    sg::LaunchFn fn = nullptr;
    if (pl.mode == 5)
        fn = sg::launcher_decoded(out_dtype);
    else if (pl.mode == 6)
        fn = sg::launcher_wide(out_dtype, residual, pl.block_k == sg::BK_BYTES ? 1 : 2);
    else if (pl.mode == 4)
        fn = sg::launcher_panel(out_dtype, residual, pl.block_k == sg::BK_BYTES ? 1 : 2);
    else if (pl.block_k == sg::BK_BYTES)  // 8-bit operands
        fn = residual ? sg::launcher_fp8_res(pl.bn, out_dtype, pl.mode) : sg::launcher_fp8_plain(pl.bn, out_dtype, pl.mode);
    else if (pl.mode == 1)
        fn = residual ? sg::launcher_res_single(pl.bn, out_dtype) : sg::launcher_plain_single(pl.bn, out_dtype);
    else
        fn = residual ? sg::launcher_res_pair(pl.bn, out_dtype, pl.mode)
                      : sg::launcher_plain_pair(pl.bn, out_dtype, pl.mode);
    if (!fn) return SG_ERR_ARG;
    const int bi = pl.bn == 128 ? 0 : pl.bn == 192 ? 1 : 2;
    sg::LaunchArgs a;
    a.ta = &ta;
    a.tb = &tb;
    a.tc = &tc;
    a.tr = &tr;
    a.prm = &prm;
    a.grid = pl.grid;
    a.smem = pl.smem;
    a.smem_optin = st.smem_optin;
    a.stream = stream;
    a.mu = &g_mu;
    const int e8 = pl.block_k == sg::BK_BYTES ? 1 : 0;
    a.attr_done = &st.attr_done[e8][bi][out_dtype][pl.mode - 1][residual ? 1 : 0];
    a.max_clusters = &st.max_clusters[e8][bi][out_dtype][pl.mode - 1][residual ? 1 : 0];
    return fn(a) == 0 ? SG_OK : SG_ERR_CUDA;
}

void fill_info(const Plan& pl, sg_plan_info* info) {
    std::memset(info, 0, sizeof(*info));
    info->block_m = sg::BM;
    info->block_n = pl.tw;
    info->block_k = static_cast<int32_t>(pl.block_k);
    info->stages = pl.stages;
    info->max_stages = pl.max_stages;
    info->tiles = static_cast<int32_t>(pl.tiles);
    info->grid = pl.grid;
    info->threads = sg::NUM_THREADS;
    info->smem_bytes = pl.smem;
    info->tmem_columns = pl.tmem_cols;
    info->tma_store = pl.tma_store;
    info->cluster_m = pl.cm;
    info->pair_mma = (pl.mode == 3 || pl.mode == 6) ? 1 : 0;
    info->group_m = pl.group_m;
    info->mode = pl.mode;
    info->ring_group = pl.ring_group;
    info->tail_units = static_cast<int32_t>(pl.units - pl.full_units);
}

bool c_tma_legal(const void* C, int64_t M, int64_t ldc, int out_dtype) {
    return (reinterpret_cast<uintptr_t>(C) & 15) == 0 && (M == 1 || (ldc * elem_bytes(out_dtype)) % 16 == 0);
}

int current_device() {
    int dev = 0;
    return cudaGetDevice(&dev) == cudaSuccess ? dev : -1;
}

// The tuned configuration for this problem, if sg_tune measured one.
bool lookup_tuned(int64_t M, int64_t N, int64_t K, int in_dtype, int out_dtype, int epi, bool a_tma, bool b_tma,
                  bool c_tma, Choice* out) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_tuned.empty()) return false;
    auto it = g_tuned.find(tune_key(current_device(), M, N, K, in_dtype, out_dtype, epi, a_tma, b_tma, c_tma));
    if (it == g_tuned.end()) return false;
    *out = it->second;
    return true;
}

// A plan gives what a strict choice asked for.
bool honours(const Plan& pl, const Choice& c) {
    return (!c.bn || pl.tw == c.bn) && (!c.mode || pl.mode == c.mode);
}

// Plan, build the tensor maps and kernel parameters, and launch (shared by
// the entry points; `st` supplies the device's attributes and status word).
// With Bq (mode 5) B is int8 codes with per-column scales b_scale, decoded
// into the resident panel; B is then unused.
int plan_and_launch_impl(DevState& st, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                    int64_t ldb, void* C, int64_t ldc, int in_dtype, int out_dtype, int epilogue, const float* bias,
                    int stages, int64_t skip_load, cudaStream_t stream, const Choice* forced = nullptr,
                    Plan* used = nullptr, const void* R = nullptr, int64_t ldr = 0, const int8_t* Bq = nullptr,
                    const float* b_scale = nullptr) {
    const int esz = elem_bytes(in_dtype);
    const bool decode = Bq != nullptr;
    const bool a_tma = (decode && K == 0) || tma_legal(A, M, lda, esz);  // mode 5 with K = 0 reads no A
    const bool b_tma = decode || tma_legal(B, K, ldb, esz);
    Choice tuned;
    const Choice* choice = forced;
    if (!choice && !decode &&
        lookup_tuned(M, N, K, in_dtype, out_dtype, epilogue, a_tma, b_tma, c_tma_legal(C, M, ldc, out_dtype), &tuned))
        choice = &tuned;
    Plan pl;
    int rc = make_plan(st, M, N, K, in_dtype, out_dtype, C, ldc, stages, a_tma, b_tma, &pl, choice, decode, R != nullptr,
                       epilogue == SG_EPI_BIAS_RELU);
    if (rc != SG_OK) return rc;
    if (choice && choice->strict && !honours(pl, *choice)) return SG_ERR_CONFIG;
    if (used) *used = pl;

    alignas(64) CUtensorMap ta, tb, tc, tr;
    std::memset(&ta, 0, sizeof(ta));
    std::memset(&tb, 0, sizeof(tb));
    std::memset(&tc, 0, sizeof(tc));
    std::memset(&tr, 0, sizeof(tr));
    if (K > 0) {
        const uint32_t kb = sg::BK_BYTES / esz, boxc = 128 / esz;
        if (a_tma && (rc = encode_2d(&ta, in_dtype, A, K, M, lda * esz, kb, sg::BM)) != SG_OK) return rc;
        if (!decode && b_tma && (rc = encode_2d(&tb, in_dtype, B, N, K, ldb * esz, boxc, kb)) != SG_OK) return rc;
    }
    const int oes = elem_bytes(out_dtype);
    if (pl.tma_store) {
        if ((rc = encode_2d(&tc, out_dtype, C, N, M, ldc * oes, 128 / oes, 32)) != SG_OK) return rc;
    }
    // a residual box has the shape of an output box (32 rows x 128 bytes)
    const bool r_tma = R != nullptr && c_tma_legal(R, M, ldr, out_dtype);
    if (r_tma && (rc = encode_2d(&tr, out_dtype, R, N, M, ldr * oes, 128 / oes, 32)) != SG_OK) return rc;

    sg::Params prm;
    std::memset(&prm, 0, sizeof(prm));
    prm.M = static_cast<int32_t>(M);
    prm.N = static_cast<int32_t>(N);
    prm.K = static_cast<int32_t>(K);
    prm.m_blocks = static_cast<int32_t>(pl.m_blocks);
    prm.n_blocks = static_cast<int32_t>(pl.n_blocks);
    prm.num_tiles = static_cast<int32_t>(pl.units);
    prm.full_units = static_cast<int32_t>(pl.full_units);
    prm.k_chunks = static_cast<int32_t>(pl.k_chunks);
    prm.stages = pl.stages;
    prm.ring_group = pl.ring_group;
    prm.group_m = pl.group_m;
    const int mma_m = (pl.mode == 3 || pl.mode == 6) ? 2 * sg::BM : sg::BM;
    prm.idesc = esz == 1 ? sg::idesc_e4m3(mma_m, pl.bn, true)
                         : sg::idesc_f16(in_dtype == SG_BF16, mma_m, pl.bn, true);
    prm.idesc_half = esz == 1 ? sg::idesc_e4m3(mma_m, pl.bn / 2, true)
                              : sg::idesc_f16(in_dtype == SG_BF16, mma_m, pl.bn / 2, true);
    prm.epi = epilogue;
    prm.tma_store = pl.tma_store;
    prm.bias = bias;
    prm.C = C;
    prm.ldc = ldc;
    prm.status = st.status;
    prm.wait_limit_ns = g_wait_limit_ns.load();
    prm.skip_load = skip_load;
    prm.a_tma = pl.a_tma;
    prm.b_tma = pl.b_tma;
    prm.A = static_cast<const uint16_t*>(A);
    prm.B = static_cast<const uint16_t*>(B);
    prm.lda = lda;
    prm.ldb = ldb;
    prm.R = R;
    prm.ldr = ldr;
    prm.r_tma = r_tma ? 1 : 0;
    prm.Bq = Bq;
    prm.b_scale = b_scale;
    prm.in_bf16 = in_dtype == SG_BF16 ? 1 : 0;
    return launch_plan(st, out_dtype, pl, ta, tb, tc, tr, prm, R != nullptr, stream);
}

// As plan_and_launch_impl, but an operand or a residual without a TMA-legal
// layout (a base off a 16-byte boundary or a pitch that is not a multiple of
// 16 bytes) is first copied, on the stream, into one stream-ordered buffer
// with 16-byte row pitches, so the kernel stages it by TMA rather than by
// element loads (on GB300, 100000 x 128 x 500 with a 500-column B: 475 us by
// element loads, 48 us copied); such a C is computed into the buffer and its
// N columns copied out row by row afterwards (its padding is not written).
// The copies move values only, so C keeps its bits.  Without the buffer (an
// allocation that fails) the kernel takes the element paths.  The
// allocation-free entry point calls the impl directly.
int plan_and_launch(DevState& st, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                    int64_t ldb, void* C, int64_t ldc, int in_dtype, int out_dtype, int epilogue, const float* bias,
                    int stages, int64_t skip_load, cudaStream_t stream, const Choice* forced = nullptr,
                    Plan* used = nullptr, const void* R = nullptr, int64_t ldr = 0, const int8_t* Bq = nullptr,
                    const float* b_scale = nullptr) {
    const int esz = elem_bytes(in_dtype), oes = elem_bytes(out_dtype);
    const bool decode = Bq != nullptr;
    const bool fix_a = K > 0 && !tma_legal(A, M, lda, esz);
    const bool fix_b = K > 0 && !decode && !tma_legal(B, K, ldb, esz);
    const bool fix_r = R != nullptr && !c_tma_legal(R, M, ldr, out_dtype);
    const bool fix_c = !c_tma_legal(C, M, ldc, out_dtype);
    auto direct = [&] {
        return plan_and_launch_impl(st, M, N, K, A, lda, B, ldb, C, ldc, in_dtype, out_dtype, epilogue, bias, stages,
                                    skip_load, stream, forced, used, R, ldr, Bq, b_scale);
    };
    if ((!fix_a && !fix_b && !fix_r && !fix_c) || !g_repack.load()) return direct();
    auto pitch16 = [](int64_t cols, int e) { return cdiv(std::max<int64_t>(cols, 1), 16 / e) * (16 / e); };
    auto up = [](uint64_t b) { return (b + 255) & ~uint64_t(255); };
    const int64_t pa = fix_a ? pitch16(K, esz) : lda, pb = fix_b ? pitch16(N, esz) : ldb;
    const int64_t pr = fix_r ? pitch16(N, oes) : ldr, pc = fix_c ? pitch16(N, oes) : ldc;
    const uint64_t a_bytes = fix_a ? up(uint64_t(M) * pa * esz) : 0, b_bytes = fix_b ? up(uint64_t(K) * pb * esz) : 0;
    const uint64_t r_bytes = fix_r ? up(uint64_t(M) * pr * oes) : 0, c_bytes = fix_c ? up(uint64_t(M) * pc * oes) : 0;
    char* buf = nullptr;
    if (pool_alloc(st, reinterpret_cast<void**>(&buf), a_bytes + b_bytes + r_bytes + c_bytes, stream) != cudaSuccess) {
        cudaGetLastError();  // no buffer: the element path
        return direct();
    }
    const auto D2D = cudaMemcpyDeviceToDevice;
    const void* A2 = fix_a ? buf : A;
    const void* B2 = fix_b ? buf + a_bytes : B;
    const void* R2 = fix_r ? buf + a_bytes + b_bytes : R;
    void* C2 = fix_c ? buf + a_bytes + b_bytes + r_bytes : C;
    bool ok = true;
    if (fix_a) ok = cudaMemcpy2DAsync(buf, pa * esz, A, lda * esz, K * esz, M, D2D, stream) == cudaSuccess;
    if (ok && fix_b)
        ok = cudaMemcpy2DAsync(buf + a_bytes, pb * esz, B, ldb * esz, N * esz, K, D2D, stream) == cudaSuccess;
    if (ok && fix_r)
        ok = cudaMemcpy2DAsync(buf + a_bytes + b_bytes, pr * oes, R, ldr * oes, N * oes, M, D2D, stream) ==
             cudaSuccess;
    int rc;
    if (ok) {
        rc = plan_and_launch_impl(st, M, N, K, A2, pa, B2, pb, C2, pc, in_dtype, out_dtype, epilogue, bias, stages,
                                  skip_load, stream, forced, used, R2, pr, Bq, b_scale);
        if (rc == SG_OK && fix_c &&
            cudaMemcpy2DAsync(C, ldc * oes, C2, pc * oes, N * oes, M, D2D, stream) != cudaSuccess)
            rc = SG_ERR_CUDA;
    } else {
        cudaGetLastError();
        rc = direct();
    }
    // released on the stream, after the kernel that reads it
    const bool freed = cudaFreeAsync(buf, stream) == cudaSuccess;
    return (rc == SG_OK && !freed) ? SG_ERR_CUDA : rc;
}

}  // namespace

extern "C" {

int sg_gemm(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
            int64_t ldc, int in_dtype, int out_dtype, int epilogue, const float* bias, int stages, void* stream) {
    int rc = check_args(M, N, K, A, lda, B, ldb, C, ldc, in_dtype, out_dtype, epilogue, bias, stages);
    if (rc != SG_OK) return rc;
    if (M == 0 || N == 0) return SG_OK;
    DevState* st = nullptr;
    if ((rc = device_state(&st)) != SG_OK) return rc;
    return plan_and_launch(*st, M, N, K, A, lda, B, ldb, C, ldc, in_dtype, out_dtype, epilogue, bias, stages,
                           g_skip_load.load(), static_cast<cudaStream_t>(stream));
}

int sg_gemm_residual(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
                     const void* R, int64_t ldr, void* C, int64_t ldc, int in_dtype, int out_dtype, int epilogue,
                     const float* bias, int stages, void* stream) {
    int rc = check_args(M, N, K, A, lda, B, ldb, C, ldc, in_dtype, out_dtype, epilogue, bias, stages);
    if (rc != SG_OK) return rc;
    if (M == 0 || N == 0) return SG_OK;
    if ((rc = check_residual(M, N, R, ldr, C, ldc, out_dtype)) != SG_OK) return rc;
    DevState* st = nullptr;
    if ((rc = device_state(&st)) != SG_OK) return rc;
    return plan_and_launch(*st, M, N, K, A, lda, B, ldb, C, ldc, in_dtype, out_dtype, epilogue, bias, stages,
                           g_skip_load.load(), static_cast<cudaStream_t>(stream), nullptr, nullptr, R, ldr);
}

int sg_gemm_qb(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const int8_t* Bq, int64_t ldb,
               const float* b_scale, void* C, int64_t ldc, int in_dtype, int out_dtype, int epilogue,
               const float* bias, int stages, void* stream) {
    if (in_dtype != SG_F16 && in_dtype != SG_BF16) return SG_ERR_DTYPE;
    // A's checks (B's are taken below: its elements are single bytes)
    int rc = check_args(M, N, K, A, lda, A, N, C, ldc, in_dtype, out_dtype, epilogue, bias, stages);
    if (rc != SG_OK) return rc;
    if (M == 0 || N == 0) return SG_OK;
    if (!b_scale || ldb > 0x7FFFFFFF) return SG_ERR_ARG;
    if (reinterpret_cast<uintptr_t>(b_scale) & 3u) return SG_ERR_ALIGN;
    if (K > 0 && (!Bq || ldb < N)) return SG_ERR_ARG;
    const uint64_t c_span = span_bytes(M, N, ldc, elem_bytes(out_dtype));
    if ((K > 0 && overlap(C, c_span, Bq, span_bytes(K, N, ldb, 1))) ||
        overlap(C, c_span, b_scale, static_cast<uint64_t>(N) * 4))
        return SG_ERR_ALIAS;
    DevState* st = nullptr;
    if ((rc = device_state(&st)) != SG_OK) return rc;
    // a K = 0 product reads no codes: any non-null pointer marks the mode
    const int8_t* codes = K > 0 ? Bq : reinterpret_cast<const int8_t*>(b_scale);
    return plan_and_launch(*st, M, N, K, A, lda, nullptr, ldb, C, ldc, in_dtype, out_dtype, epilogue, bias, stages,
                           g_skip_load.load(), static_cast<cudaStream_t>(stream), nullptr, nullptr, nullptr, 0, codes,
                           b_scale);
}

int sg_gemm_host(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
                 const void* R, int64_t ldr, void* C, int64_t ldc, int in_dtype, int out_dtype, int epilogue,
                 const float* bias, int stages, void* stream) {
    int rc = check_args(M, N, K, A, lda, B, ldb, C, ldc, in_dtype, out_dtype, epilogue, bias, stages);
    if (rc != SG_OK) return rc;
    if (M == 0 || N == 0) return SG_OK;
    const int esz = elem_bytes(in_dtype), oes = elem_bytes(out_dtype);
    if (R && (rc = check_residual(M, N, R, ldr, C, ldc, out_dtype)) != SG_OK) return rc;
    DevState* st = nullptr;
    if ((rc = device_state(&st)) != SG_OK) return rc;
    if ((rc = host_streams(*st)) != SG_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    // Device copies keep the host pitch when it is a whole number of 16-byte
    // units (each chunk then moves as one contiguous span of the host
    // operand; the padding columns it carries are never read); otherwise the
    // rows are packed to a 16-byte pitch by a 2-D copy.  Every operand and
    // every row chunk of it is then TMA-legal.  C returns as one span only
    // when it has no padding columns, so the caller's padding is never
    // written.
    auto dev_pitch = [](int64_t ld, int64_t cols, int e) {
        return (ld * e) % 16 == 0 ? ld : cdiv(std::max<int64_t>(cols, 1), 16 / e) * (16 / e);
    };
    auto up = [](uint64_t b) { return (b + 255) & ~uint64_t(255); };
    const int64_t pa = dev_pitch(lda, K, esz), pb = dev_pitch(ldb, N, esz), pc = dev_pitch(ldc, N, oes);
    const int64_t pr = R ? dev_pitch(ldr, N, oes) : 0;
    const uint64_t a_bytes = K > 0 ? up(uint64_t(M) * pa * esz) : 0;
    const uint64_t b_bytes = K > 0 ? up(uint64_t(K) * pb * esz) : 0;
    const uint64_t c_bytes = up(uint64_t(M) * pc * oes);
    const uint64_t r_bytes = R ? up(uint64_t(M) * pr * oes) : 0;
    const uint64_t bias_bytes = bias ? up(uint64_t(N) * 4) : 0;
    const uint64_t total = a_bytes + b_bytes + c_bytes + r_bytes + bias_bytes;
    const uint64_t copy_bytes = uint64_t(M) * K * esz + uint64_t(K) * N * esz + uint64_t(M) * N * oes * (R ? 2 : 1);
    const int64_t chunk = host_chunk_rows(M, copy_bytes);

    std::lock_guard<std::mutex> lk(g_host_mu);
    char* buf = nullptr;
    if (pool_alloc(*st, reinterpret_cast<void**>(&buf), total, s) != cudaSuccess) return SG_ERR_CUDA;
    char* dA = K > 0 ? buf : nullptr;
    char* dB = K > 0 ? buf + a_bytes : nullptr;
    char* dC = buf + a_bytes + b_bytes;
    char* dR = R ? dC + c_bytes : nullptr;
    float* dbias = bias ? reinterpret_cast<float*>(dC + c_bytes + r_bytes) : nullptr;
    const char* hA = static_cast<const char*>(A);
    const char* hR = static_cast<const char*>(R);
    char* hC = static_cast<char*>(C);
    // rows [r0, r0 + rows) of a cols-wide operand between pitches hp and dp
    auto copy_rows = [&](void* dst, int64_t dp, const void* src, int64_t hp, int64_t cols, int e, int64_t rows,
                         cudaMemcpyKind kind, cudaStream_t on, bool span_ok) {
        const int64_t sp = kind == cudaMemcpyHostToDevice ? hp : dp, tp = kind == cudaMemcpyHostToDevice ? dp : hp;
        if (span_ok && sp == tp)
            return cudaMemcpyAsync(dst, src, span_bytes(rows, cols, sp, e), kind, on) == cudaSuccess;
        return cudaMemcpy2DAsync(dst, tp * e, src, sp * e, cols * e, rows, kind, on) == cudaSuccess;
    };
    const auto H2D = cudaMemcpyHostToDevice, D2H = cudaMemcpyDeviceToHost;

    // fork: the copy streams start after the work already on `stream`
    bool ok = cudaEventRecord(st->ev_fork, s) == cudaSuccess &&
              cudaStreamWaitEvent(st->h2d, st->ev_fork, 0) == cudaSuccess &&
              cudaStreamWaitEvent(st->d2h, st->ev_fork, 0) == cudaSuccess &&
              cudaStreamWaitEvent(st->comp, st->ev_fork, 0) == cudaSuccess;
    if (ok && bias) ok = cudaMemcpyAsync(dbias, bias, size_t(N) * 4, H2D, st->h2d) == cudaSuccess;
    if (ok && K > 0) ok = copy_rows(dB, pb, B, ldb, N, esz, K, H2D, st->h2d, true);
    // Chunks alternate between `stream` and the library's second compute
    // stream, so a chunk's CTAs take SMs as the previous chunk's last wave
    // leaves them (one CTA per SM either way: each holds more than half the
    // shared memory and all of the tensor memory).
    int gemm_rc = SG_OK;
    int64_t idx = 0;
    for (int64_t r0 = 0; ok && r0 < M; r0 += chunk, ++idx) {
        const int64_t rows = std::min(chunk, M - r0);
        cudaStream_t cs = (idx % 2 == 0) ? s : st->comp;
        if (K > 0) ok = copy_rows(dA + r0 * pa * esz, pa, hA + r0 * lda * esz, lda, K, esz, rows, H2D, st->h2d, true);
        if (ok && R)
            ok = copy_rows(dR + r0 * pr * oes, pr, hR + r0 * ldr * oes, ldr, N, oes, rows, H2D, st->h2d, true);
        ok = ok && cudaEventRecord(st->ev_in, st->h2d) == cudaSuccess &&
             cudaStreamWaitEvent(cs, st->ev_in, 0) == cudaSuccess;
        if (!ok) break;
        gemm_rc = plan_and_launch(*st, rows, N, K, K > 0 ? dA + r0 * pa * esz : nullptr, pa, dB, pb,
                                  dC + r0 * pc * oes, pc, in_dtype, out_dtype, epilogue, dbias, stages,
                                  g_skip_load.load(), cs, nullptr, nullptr, R ? dR + r0 * pr * oes : nullptr, pr);
        if (gemm_rc != SG_OK) break;
        ok = cudaEventRecord(st->ev_gemm, cs) == cudaSuccess &&
             cudaStreamWaitEvent(st->d2h, st->ev_gemm, 0) == cudaSuccess &&
             copy_rows(hC + r0 * ldc * oes, pc, dC + r0 * pc * oes, ldc, N, oes, rows, D2H, st->d2h, ldc == N);
    }
    // join (also after a failure, so nothing queued outlives the buffer):
    // `stream` waits for both copy streams, then releases the buffer
    bool joined = cudaEventRecord(st->ev_out, st->d2h) == cudaSuccess &&
                  cudaStreamWaitEvent(s, st->ev_out, 0) == cudaSuccess &&
                  cudaEventRecord(st->ev_in, st->h2d) == cudaSuccess &&
                  cudaStreamWaitEvent(s, st->ev_in, 0) == cudaSuccess &&
                  cudaEventRecord(st->ev_comp, st->comp) == cudaSuccess &&
                  cudaStreamWaitEvent(s, st->ev_comp, 0) == cudaSuccess;
    if (!joined) {
        cudaStreamSynchronize(st->d2h);
        cudaStreamSynchronize(st->h2d);
        cudaStreamSynchronize(st->comp);
    }
    const bool freed = cudaFreeAsync(buf, s) == cudaSuccess;
    if (gemm_rc != SG_OK) return gemm_rc;
    return (ok && joined && freed) ? SG_OK : SG_ERR_CUDA;
}

int sg_plan(int64_t M, int64_t N, int64_t K, int in_dtype, int out_dtype, int epilogue, int stages, int64_t ldc,
            const void* C, sg_plan_info* info) {
    if (!info) return SG_ERR_ARG;
    if (!valid_in(in_dtype) || !valid_out(out_dtype) || !valid_epi(epilogue)) return SG_ERR_DTYPE;
    if (M < 0 || N < 0 || K < 0 || ldc < N) return SG_ERR_ARG;
    if (stages < 0 || stages > SG_MAX_STAGES) return SG_ERR_STAGES;
    std::memset(info, 0, sizeof(*info));
    DevState* st = nullptr;
    int rc = device_state(&st);
    if (rc != SG_OK) return rc;
    Plan pl;
    Choice tuned;
    const bool have = lookup_tuned(M, N, K, in_dtype, out_dtype, epilogue, true, true,
                                   c_tma_legal(C, M, ldc, out_dtype), &tuned);
    if ((rc = make_plan(*st, M, N, K, in_dtype, out_dtype, C, ldc, stages, true, true, &pl, have ? &tuned : nullptr,
                        false, false, epilogue == SG_EPI_BIAS_RELU)) != SG_OK)
        return rc;
    fill_info(pl, info);
    return SG_OK;
}

// The launch configuration an sg_config asks for, validated on the host.
static int config_choice(const sg_config* cfg, Choice* c, int* stages) {
    const sg_config z = {};
    const sg_config& g = cfg ? *cfg : z;
    if (g.block_n != 0 && !valid_tile(g.block_n)) return SG_ERR_CONFIG;
    if (g.mode != 0 && !valid_mode(g.mode)) return SG_ERR_CONFIG;
    if (g.group_m < 0 || g.group_m > 64 || g.tail_split < -1 || g.tail_split > 1) return SG_ERR_CONFIG;
    if (g.stages < 0 || g.stages > SG_MAX_STAGES) return SG_ERR_STAGES;
    c->bn = g.block_n;
    c->mode = g.mode;
    c->group_m = g.group_m;
    c->tail_split = g.tail_split;
    c->strict = true;
    *stages = g.stages;
    // all zeros: exactly sg_gemm (a tuned configuration still applies)
    return (g.block_n || g.mode || g.group_m || g.tail_split) ? 1 : 0;
}

int sg_gemm_ex(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
               const void* R, int64_t ldr, void* C, int64_t ldc, int in_dtype, int out_dtype, int epilogue,
               const float* bias, const sg_config* config, void* stream) {
    Choice c;
    int stages = 0;
    const int given = config_choice(config, &c, &stages);
    if (given < 0) return given;
    int rc = check_args(M, N, K, A, lda, B, ldb, C, ldc, in_dtype, out_dtype, epilogue, bias, stages);
    if (rc != SG_OK) return rc;
    if (M == 0 || N == 0) return SG_OK;
    if (R && (rc = check_residual(M, N, R, ldr, C, ldc, out_dtype)) != SG_OK) return rc;
    DevState* st = nullptr;
    if ((rc = device_state(&st)) != SG_OK) return rc;
    return plan_and_launch(*st, M, N, K, A, lda, B, ldb, C, ldc, in_dtype, out_dtype, epilogue, bias, stages,
                           g_skip_load.load(), static_cast<cudaStream_t>(stream), given ? &c : nullptr, nullptr, R,
                           R ? ldr : 0);
}

int sg_plan_ex(int64_t M, int64_t N, int64_t K, int in_dtype, int out_dtype, int epilogue, int64_t ldc,
               const void* C, const sg_config* config, sg_plan_info* info) {
    if (!info) return SG_ERR_ARG;
    std::memset(info, 0, sizeof(*info));
    Choice c;
    int stages = 0;
    const int given = config_choice(config, &c, &stages);
    if (given < 0) return given;
    if (!valid_in(in_dtype) || !valid_out(out_dtype) || !valid_epi(epilogue)) return SG_ERR_DTYPE;
    if (M < 0 || N < 0 || K < 0 || ldc < N) return SG_ERR_ARG;
    DevState* st = nullptr;
    int rc = device_state(&st);
    if (rc != SG_OK) return rc;
    Choice tuned;
    const Choice* choice = given ? &c : nullptr;
    if (!choice && lookup_tuned(M, N, K, in_dtype, out_dtype, epilogue, true, true, c_tma_legal(C, M, ldc, out_dtype),
                                &tuned))
        choice = &tuned;
    Plan pl;
    if ((rc = make_plan(*st, M, N, K, in_dtype, out_dtype, C, ldc, stages, true, true, &pl, choice, false, false,
                        epilogue == SG_EPI_BIAS_RELU)) != SG_OK)
        return rc;
    if (given && !honours(pl, c)) return SG_ERR_CONFIG;
    fill_info(pl, info);
    return SG_OK;
}

int sg_tune(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
            int64_t ldc, int in_dtype, int out_dtype, int epilogue, const float* bias, void* stream,
            sg_plan_info* best, float* best_ms) {
    int rc = check_args(M, N, K, A, lda, B, ldb, C, ldc, in_dtype, out_dtype, epilogue, bias, 0);
    if (rc != SG_OK) return rc;
    if (M == 0 || N == 0) return SG_OK;
    DevState* st = nullptr;
    if ((rc = device_state(&st)) != SG_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int esz = elem_bytes(in_dtype);
    const bool a_tma = tma_legal(A, M, lda, esz), b_tma = tma_legal(B, K, ldb, esz);
    const bool c_tma = c_tma_legal(C, M, ldc, out_dtype);
    const int64_t m_blocks = cdiv(M, sg::BM);

    // the configurations that fit this problem
    std::vector<Choice> cands;
    for (int bn : {128, 192, 256}) {
        if (bn % (128 / esz)) continue;  // whole 128-byte B boxes
        if (bn > 128 && N <= bn - 64) continue;  // a tile mostly past N
        for (int mode : {1, 3}) {
            if (mode == 3 && ((bn / (128 / esz)) % 2 != 0 || m_blocks < 2 || !a_tma || !b_tma)) continue;
            for (int g : {4, 8, 12, 16}) {
                Choice c;
                c.bn = bn;
                c.mode = mode;
                c.group_m = g;
                // the raster only matters when there are more tiles than CTAs
                if (g != 12 && m_blocks * cdiv(N, bn) <= st->sm_count) continue;
                cands.push_back(c);
            }
        }
        if (bn == 128 && a_tma && b_tma) {  // resident B, when it fits (the planner checks)
            Choice c;
            c.bn = 128;
            c.mode = 4;
            cands.push_back(c);
        }
    }
    if (a_tma && b_tma && m_blocks >= 2 && N > 256) {  // wide paired tiles (two 256-column accumulators)
        for (int g : {8, 12, 16}) {
            Choice c;
            c.bn = 512;
            c.mode = 6;
            c.group_m = g;
            if (g != 12 && m_blocks * cdiv(N, 512) <= st->sm_count) continue;
            cands.push_back(c);
        }
    }
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) return SG_ERR_CUDA;
    float best_t = -1.0f;
    Choice best_c;
    Plan best_p;
    constexpr int kReps = 3;
    for (const Choice& c : cands) {
        Plan pl;
        // one untimed run (sets kernel attributes, warms caches), then the reps
        rc = plan_and_launch(*st, M, N, K, A, lda, B, ldb, C, ldc, in_dtype, out_dtype, epilogue, bias, 0, -1, s, &c,
                             &pl);
        if (rc != SG_OK) continue;
        float t_min = -1.0f;
        for (int r = 0; r < kReps && rc == SG_OK; ++r) {
            if (cudaEventRecord(e0, s) != cudaSuccess) rc = SG_ERR_CUDA;
            if (rc == SG_OK)
                rc = plan_and_launch(*st, M, N, K, A, lda, B, ldb, C, ldc, in_dtype, out_dtype, epilogue, bias, 0, -1,
                                     s, &c);
            if (rc == SG_OK && cudaEventRecord(e1, s) != cudaSuccess) rc = SG_ERR_CUDA;
            if (rc == SG_OK && cudaEventSynchronize(e1) != cudaSuccess) rc = SG_ERR_CUDA;
            float ms = 0.0f;
            if (rc == SG_OK && cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess) rc = SG_ERR_CUDA;
            if (rc == SG_OK && (t_min < 0.0f || ms < t_min)) t_min = ms;
        }
        if (rc != SG_OK) break;
        if (best_t < 0.0f || t_min < best_t) {
            best_t = t_min;
            best_c = c;
            best_p = pl;
        }
    }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (rc != SG_OK) return rc;
    if (best_t < 0.0f) return SG_ERR_STAGES;  // nothing fitted
    best_c.stages = best_p.stages;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        g_tuned[tune_key(current_device(), M, N, K, in_dtype, out_dtype, epilogue, a_tma, b_tma, c_tma)] = best_c;
    }
    if (best) fill_info(best_p, best);
    if (best_ms) *best_ms = best_t;
    return SG_OK;
}

int sg_tune_clear(void) {
    std::lock_guard<std::mutex> lk(g_mu);
    const int n = static_cast<int>(g_tuned.size());
    g_tuned.clear();
    return n;
}

int sg_tune_count(void) {
    std::lock_guard<std::mutex> lk(g_mu);
    return static_cast<int>(g_tuned.size());
}

int sg_device_status(void* stream) {
    DevState* st = nullptr;
    int rc = device_state(&st);
    if (rc != SG_OK) return rc;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return SG_ERR_CUDA;
    int h = 0;
    if (cudaMemcpy(&h, st->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return SG_ERR_CUDA;
    if (h != 0) {
        if (cudaMemset(st->status, 0, sizeof(int)) != cudaSuccess) return SG_ERR_CUDA;
        return SG_ERR_TIMEOUT;
    }
    return SG_OK;
}

void sg_set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns.store(ns ? ns : 1); }

uint64_t sg_get_wait_limit_ns(void) { return g_wait_limit_ns.load(); }

const char* sg_strerror(int code) {
    switch (code) {
        case SG_OK: return "success";
        case SG_ERR_ARG: return "invalid argument (size, leading dimension, pointer or bias)";
        case SG_ERR_DTYPE: return "unsupported storage type or epilogue";
        case SG_ERR_STAGES: return "stage count out of range or does not fit in shared memory";
        case SG_ERR_ALIAS: return "C overlaps A, B, R or bias";
        case SG_ERR_ALIGN: return "an operand, C, R, bias or scale base not aligned to its element size";
        case SG_ERR_ARCH: return "current device is not sm_103 (GB300)";
        case SG_ERR_CUDA: return "CUDA runtime or driver error";
        case SG_ERR_TIMEOUT: return "a device-side wait gave up";
        case SG_ERR_CONFIG: return "the requested launch configuration does not fit this problem";
        default: return "unknown error code";
    }
}

int sg_version(void) { return SG_VERSION; }

// Test hook, deliberately absent from the public header: launches after this
// call never copy the K chunk with global index `it` (-1 restores normal
// operation), so the MMA warp's bounded wait for it runs out.
int sg_test_set_skip_load(int64_t it) {
    g_skip_load.store(it < 0 ? -1 : it);
    return SG_OK;
}

int sg_test_set_tile_n(int bn) {
    if (bn != 0 && !valid_bn(bn)) return SG_ERR_ARG;
    g_force_bn.store(bn);
    return SG_OK;
}

int sg_test_set_cluster(int mode) {
    if (mode != 0 && !valid_mode(mode)) return SG_ERR_ARG;
    g_force_mode.store(mode);
    return SG_OK;
}

int sg_test_set_tail_split(int on) {
    if (on != 0 && on != 1) return SG_ERR_ARG;
    g_tail_split.store(on);
    return SG_OK;
}

int sg_test_set_repack(int on) {
    if (on != 0 && on != 1) return SG_ERR_ARG;
    g_repack.store(on);
    return SG_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free entry point (sg_gemm_noalloc): the status word lives in a
// static device array instead of library-allocated memory.

static __device__ __align__(256) int sg_noalloc_scratch[SG_NOALLOC_SCRATCH_BYTES / sizeof(int)];

namespace {

constexpr size_t kNoallocScratchNeed = sizeof(int);  // one status word, whatever the problem size
DevState g_noalloc_dev[kMaxDevices];

// Per-device set-up for the allocation-free path: attributes, the tensor-map
// encoder and the device address of the static scratch array.  No
// allocation.  Runs on the first call on each device.
int noalloc_state(DevState** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SG_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    DevState& st = g_noalloc_dev[dev];
    if (!st.ready) {
        if (cudaDeviceGetAttribute(&st.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&st.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return SG_ERR_CUDA;
        if (st.major != 10 || st.minor != 3) return SG_ERR_ARCH;
        if (cudaDeviceGetAttribute(&st.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&st.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&st.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) !=
                cudaSuccess)
            return SG_ERR_CUDA;
        if (int rc = ensure_encode_fn(); rc != SG_OK) return rc;
        // In host code the array's name is only a host-side stand-in; the
        // kernel must be given the device address.
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, sg_noalloc_scratch) != cudaSuccess || ptr == nullptr) return SG_ERR_CUDA;
        st.status = static_cast<int*>(ptr);
        st.ready = true;
    }
    *out = &st;
    return SG_OK;
}

}  // namespace

extern "C" {

int sg_gemm_noalloc(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
                    int64_t ldc, int in_dtype, int out_dtype, int epilogue, const float* bias, int stages,
                    void* stream) {
    static_assert(kNoallocScratchNeed <= SG_NOALLOC_SCRATCH_BYTES, "scratch array too small");
    int rc = check_args(M, N, K, A, lda, B, ldb, C, ldc, in_dtype, out_dtype, epilogue, bias, stages);
    if (rc != SG_OK) return rc;
    if (M == 0 || N == 0) return SG_OK;
    if (kNoallocScratchNeed > SG_NOALLOC_SCRATCH_BYTES) return SG_ERR_ARG;  // the need is fixed; never taken
    DevState* st = nullptr;
    if ((rc = noalloc_state(&st)) != SG_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the array keeps the previous call's word: clear it for this call
    if (cudaMemsetAsync(st->status, 0, sizeof(int), s) != cudaSuccess) return SG_ERR_CUDA;
    // the impl: an operand without a TMA-legal layout takes the element path here
    return plan_and_launch_impl(*st, M, N, K, A, lda, B, ldb, C, ldc, in_dtype, out_dtype, epilogue, bias, stages,
                                g_skip_load.load(), s);
}

int sg_gemm_noalloc_status(void* stream) {
    DevState* st = nullptr;
    int rc = noalloc_state(&st);
    if (rc != SG_OK) return rc;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return SG_ERR_CUDA;
    int h = 0;
    if (cudaMemcpy(&h, st->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return SG_ERR_CUDA;
    return h != 0 ? SG_ERR_TIMEOUT : SG_OK;
}

}  // extern "C"
