// sg_kernel.cuh -- the persistent, warp-specialised sm_103a GEMM kernel
//
//     C = epilogue(A . B [+ R]),  A: M x K row-major, B: K x N row-major
//     (fp16/bf16/FP8 E4M3, or int8 codes with per-column scales in mode 5),
//     fp32 accumulation in tensor memory, C fp32 / fp16 / bf16.
//
// Roles (one CTA per SM, 320 threads):
//   warp 0      TMA producer: copies the A tile [128 x 64] and the B tile
//               [64 x BN] of each K chunk into slot s = chunk mod stages of
//               a shared-memory ring, 128-byte swizzled.  Operand elements
//               outside M, N or K are zero-filled by the copy engine: this is
//               the "gate that copies 0 where it fails" of Tolk.Stage
//               ("operands") and the "elements past the edge read 0" of
//               gizml:tile ("In.at").
//   warp 1      allocates tensor memory; one elected thread runs the loop,
//               issuing tcgen05.mma for each filled slot into a 128 x BN
//               fp32 accumulator and freeing the slot with tcgen05.commit.
//               512 / BN (at most 4) accumulators rotate, so the epilogue of
//               earlier tiles overlaps the main loop of the next.
//   warps 2-9   epilogue: two warps per 32-lane quarter of tensor memory
//               (a warp may only read the quarter given by its index mod 4),
//               each taking every other 128-byte-wide column chunk:
//               tcgen05.ld, + bias, ReLU, one round-to-nearest-even
//               conversion, 128-byte swizzled staging in shared memory and a
//               TMA store that does not write elements outside M x N
//               (gizml:tile, "Out.put").
//
// Five modes (MODE; the numbers are those of sg_plan_info.mode):
//   1  one CTA per 128 x BN tile.
//   3  paired MMA (tcgen05 cta_group::2): the two CTAs of a cluster compute
//      one 256 x BN tile.  Each CTA stages its own 128 rows of A and its own
//      BN/2 columns of B (so a stage is 32 KiB instead of 48 KiB for
//      BN = 256 and the ring is 6 deep); one thread of the even CTA issues
//      the MMAs, whose accumulator rows live in each CTA's own tensor
//      memory.  Both CTAs' copies complete on the even CTA's full barrier;
//      its commits free the ring slots and hand accumulators to the
//      epilogues of both CTAs; both epilogues release accumulators on the
//      even CTA's barrier.
//   4  resident B ("decoded panels", Tolk.Stage): for a small K x N, each
//      CTA stages all of B once (every K chunk of every 128-column block)
//      and streams only A, one 128-row tile per ring slot; the MMAs of
//      every column block of that row tile read the one A slot, each into
//      its own rotating accumulator.  Tile units are (row tile, column
//      block) in that order; the epilogue is the same as mode 1's.
//   5  decoded panel: mode 4 with B given as int8 codes and one fp32 scale
//      per column.  At CTA start the eight epilogue warps decode all of B
//      into the resident panel, each code to the 16-bit value equal to it,
//      in the layout TMA would give (Tolk.Stage, "Decoded panels on the
//      host": the panel is decoded once and read back by every trip of the
//      other output loop); the epilogue multiplies by the column's scale,
//      fused with the bias.
//   6  wide paired tiles: mode 3 with a 256 x 2BN tile (BN = 256) held as
//      two BN-wide accumulators.  Each CTA stages its 128 rows of A once per
//      K chunk for both accumulators and its half of each accumulator's B
//      columns, so a K chunk moves 48 KiB per CTA for 128 x 512 x 64
//      products instead of 32 KiB for 128 x 256 x 64 (a quarter fewer
//      operand bytes per product).  The first accumulator goes to the
//      epilogue before the second one's last MMAs, the next tile claims its
//      second accumulator only after its first one's first MMAs are issued,
//      and the epilogue (16-bit output, no residual) hands each accumulator
//      back as soon as its values are in registers, before storing them:
//      the tile boundary waits only for those reads, which overlap MMAs.
//
// The ring generalises the two-slot pipeline of Tolk.Stage (copy chunk k+1
// into slot (k+1) mod 2 while computing on slot k mod 2) and the `stages`
// knob of gizml:tile ("Program.stages") to S slots; full/empty mbarriers with
// phase bits replace the workgroup barrier.  With 6 or 8 slots and both
// operands copied by TMA, slots are filled and consumed in pairs on the
// first slot's barriers (the MMA warp then waits once per two chunks; each
// wait stalls its issue long enough for the tensor pipe to run dry).  Every
// stage count issues the same MMAs in the same K order, so C is
// bit-identical for all of them (Tolk.Stage: staging moves values and never
// rounds them).
//
// Each warp's loop trip counts depend only on the problem size and the tile
// index (Tolk.Uniform: barriers and matrix multiply-accumulates run under
// uniform loop bounds); ragged edges are handled by zero-fill, never by
// divergent trip counts.
//
// Every wait on an mbarrier is bounded in time.  A wait that runs out sets a
// CTA-wide abort flag and the device status word; the other roles see the
// flag, leave their loops, wait (bounded) for their own copies and MMAs in
// flight, and the CTA frees its tensor memory and exits normally.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "sg_ptx.cuh"
#include "stage_gemm.h"

namespace sg {

constexpr int BM = 128;                 // tile rows = MMA M = tensor-memory lanes
// Operand geometry in bytes is the same for 16-bit (ESZ = 2) and 8-bit
// (ESZ = 1) elements: a stage holds one 128-byte swizzle row of K per A row
// (64 or 128 elements), an MMA consumes 32 bytes of K (16 or 32 elements),
// a B box is 128 bytes of N (64 or 128 columns) by the stage's K rows.
constexpr int BK_BYTES = 128;
constexpr int A_STAGE_BYTES = BM * BK_BYTES;
template <int ESZ>
struct Geom {
    static_assert(ESZ == 1 || ESZ == 2, "8- or 16-bit operands");
    static constexpr int KB = BK_BYTES / ESZ;        // K elements per stage
    static constexpr int UK = 32 / ESZ;              // K elements per MMA
    static constexpr int BOXC = 128 / ESZ;           // B columns per TMA box
    static constexpr int B_BOX_BYTES = KB * 128;     // one B box: KB rows x 128 bytes
    static constexpr int B_KSTEP_BYTES = UK * 128;   // B descriptor advance per MMA (UK rows)
};
constexpr int BK = Geom<2>::KB;  // K elements per stage for 16-bit operands
constexpr int EPI_WARPS = 8;
constexpr int NUM_THREADS = 64 + 32 * EPI_WARPS;
constexpr int EPI_BUF_BYTES = 32 * 128;     // one warp's staging buffer: 32 rows x 128 bytes
constexpr int TMEM_COLS = 512;              // the whole tensor memory of the SM
constexpr int MAX_ACC = 4;                  // accumulators in flight (512 / 128)
constexpr int SMEM_ALIGN = 1024;            // 128-byte swizzle atoms repeat every 1024 bytes
constexpr int BAR_AREA = 512;

// Device status word values: 0 = fine; otherwise a timeout site code.
constexpr int STATUS_TIMEOUT = 0x5400;
constexpr int SITE_PRODUCER_EMPTY = 1, SITE_MMA_TMEM_EMPTY = 2, SITE_MMA_FULL = 3, SITE_EPI_TMEM_FULL = 4,
              SITE_EPI_RESIDUAL = 5;

// BN: accumulator columns per tile; BL: B columns this CTA stages per K chunk
// (BN, or BN / 2 for the paired MMA).
template <int BN, int BL = BN>
struct Layout {
    static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN must be 64..256 in steps of 64");
    static_assert(BL % 64 == 0 && BL <= BN, "B is staged in whole 64-column boxes");
    // B per stage: BL columns x KB rows of ESZ bytes = BL x 128 bytes for either element size
    static constexpr int B_STAGE_BYTES = BK_BYTES * BL;
    static constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
    static constexpr int ACC = (TMEM_COLS / BN) < MAX_ACC ? (TMEM_COLS / BN) : MAX_ACC;
    static __host__ __device__ constexpr int epi_offset(int stages) { return stages * STAGE_BYTES; }
    static __host__ __device__ constexpr int bar_offset(int stages) {
        return epi_offset(stages) + EPI_WARPS * EPI_BUF_BYTES;
    }
    // dynamic shared memory to request (with slack for aligning the base)
    static __host__ __device__ constexpr int smem_bytes(int stages) { return bar_offset(stages) + BAR_AREA + SMEM_ALIGN; }
};

struct Params {
    int32_t M, N, K;
    int32_t m_blocks, n_blocks, num_tiles, k_chunks;  // num_tiles counts work units (below)
    // Work units: units below full_units are whole cluster tiles (CM row
    // blocks by BN columns) in raster order; the tiles after them, the last
    // ones of the raster, are each split into two units of BN / 2 columns
    // (their left half first) so that a short last wave spreads over twice
    // as many clusters.  Without a split full_units == num_tiles.
    int32_t full_units;
    uint32_t idesc_half;   // tcgen05 instruction descriptor of a half-width unit
    int32_t stages;
    int32_t ring_group;    // ring slots filled and consumed together on one barrier pair (1 or 2)
    int32_t group_m;       // tile raster: group_m row-blocks swept together for L2 reuse
    uint32_t idesc;        // tcgen05 instruction descriptor
    int32_t epi;           // SG_EPI_*
    int32_t tma_store;     // 1: TMA stores of C, 0: masked element stores
    const float* bias;
    void* C;
    int64_t ldc;
    int* status;
    uint64_t wait_limit_ns;
    int64_t skip_load;     // test hook: this global K-chunk index is never copied (-1: off)
    // Operands without a TMA-legal layout (base not 16-byte aligned, or a row
    // pitch that is not a multiple of 16 bytes) are copied by the producer
    // warp with element loads instead (single-CTA mode only).
    int32_t a_tma, b_tma;  // 1: copied by TMA, 0: by element loads
    const void* A;         // used when a_tma == 0
    const void* B;         // used when b_tma == 0
    int64_t lda, ldb;
    // Residual R (M x N, the output's type), added to the accumulator before
    // the bias and the ReLU; may be C itself (same address and pitch).
    const void* R;
    int64_t ldr;
    int32_t r_tma;         // 1: R tiles are loaded by TMA, 0: by element loads
    // Mode 5: B given as int8 codes (K x N, pitch ldb) with one fp32 scale
    // per column; decoded into the resident panel as the operands' 16-bit
    // type (bf16 when in_bf16), the scale applied to the accumulator.
    const int8_t* Bq;
    const float* b_scale;
    int32_t in_bf16;
};

template <int ESZ>
__device__ __forceinline__ uint32_t load_elem(const void* X, int64_t idx) {
    if constexpr (ESZ == 2) {
        return __ldg(static_cast<const uint16_t*>(X) + idx);
    } else {
        return __ldg(static_cast<const uint8_t*>(X) + idx);
    }
}

// Element-load staging of one A chunk (rows m0.., one stage of K from k0)
// into the same 128-byte-swizzled K-major layout the TMA box produces: row r
// at r * 128, 16-byte chunk c of it at c ^ (r mod 8).  Out-of-range elements
// are written as 0 (Tolk.Stage: a gate whose index fails copies 0).  Whole
// warp.
template <int ESZ>
__device__ __forceinline__ void copy_a_elements(uint32_t dst, const Params& p, int m0, int k0, int lane) {
    constexpr int EPW = 4 / ESZ;   // elements per 32-bit word
    constexpr int EPC = 16 / ESZ;  // elements per 16-byte chunk
#pragma unroll 1
    for (int c = lane; c < BM * 8; c += 32) {
        const int r = c >> 3, ch = c & 7;
        const int row = m0 + r;
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            uint32_t word = 0;
#pragma unroll
            for (int t = 0; t < EPW; ++t) {
                const int k = k0 + ch * EPC + e * EPW + t;
                if (row < p.M && k < p.K)
                    word |= load_elem<ESZ>(p.A, static_cast<int64_t>(row) * p.lda + k) << (8 * ESZ * t);
            }
            w[e] = word;
        }
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst + r * 128 + ((ch ^ (r & 7)) << 4)),
                     "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                     : "memory");
    }
}

// The same for one B chunk (one stage of K rows from k0, columns n0..n0+ncols-1)
// into the MN-major layout of the TMA boxes: 128-byte-wide box j at
// j * (box bytes), K row kr at kr * 128, 16-byte chunk c of it at c ^ (kr mod 8).
template <int ESZ>
__device__ __forceinline__ void copy_b_elements(uint32_t dst, const Params& p, int k0, int n0, int ncols, int lane) {
    using G = Geom<ESZ>;
    constexpr int EPW = 4 / ESZ;
    constexpr int EPC = 16 / ESZ;
    const int chunks = ncols / EPC;  // 16-byte chunks per K row
#pragma unroll 1
    for (int c = lane; c < G::KB * chunks; c += 32) {
        const int kr = c / chunks, cc = c - kr * chunks;
        const int j = cc >> 3, ch = cc & 7;
        const int k = k0 + kr;
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            uint32_t word = 0;
#pragma unroll
            for (int t = 0; t < EPW; ++t) {
                const int n = n0 + cc * EPC + e * EPW + t;
                if (k < p.K && n < p.N)
                    word |= load_elem<ESZ>(p.B, static_cast<int64_t>(k) * p.ldb + n) << (8 * ESZ * t);
            }
            w[e] = word;
        }
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst + j * G::B_BOX_BYTES + kr * 128 +
                                                                     ((ch ^ (kr & 7)) << 4)),
                     "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                     : "memory");
    }
}

// Linear cluster-tile index -> (row block of this CTA, column block), with a
// grouped raster over cluster row blocks (CM row blocks each): group_m of
// them are swept together for L2 reuse.  Odd groups sweep the column blocks
// backwards, so a group starts on the B columns the previous one ended on,
// which are still in L2.
template <int CM>
__device__ __forceinline__ void tile_coords(int tile, const Params& p, uint32_t rank, int& mb, int& nb) {
    const int mc_blocks = (p.m_blocks + CM - 1) / CM;
    const int per_group = p.group_m * p.n_blocks;
    const int g = tile / per_group;
    const int first_m = g * p.group_m;
    const int gsize = min(mc_blocks - first_m, p.group_m);
    const int r = tile - g * per_group;
    mb = (first_m + r % gsize) * CM + static_cast<int>(rank);
    nb = r / gsize;
    if (g & 1) nb = p.n_blocks - 1 - nb;
}

// Row block and first column of work unit `u` (modes 1, 3, 6; TW is the
// tile width); returns its width in columns.  Only 256-column tiles of
// 16-bit operands and 512-column wide tiles are ever split: each half is
// then a whole number of 128-byte B boxes in every CTA.
template <int CM, int TW, int ESZ>
__device__ __forceinline__ int unit_coords(int u, const Params& p, uint32_t rank, int& mb, int& col0) {
    constexpr bool SPLITTABLE = (TW == 256 && ESZ == 2) || TW == 512;
    int nb;
    if (!SPLITTABLE || u < p.full_units) {
        tile_coords<CM>(u, p, rank, mb, nb);
        col0 = nb * TW;
        return TW;
    }
    const int v = u - p.full_units;
    tile_coords<CM>(p.full_units + (v >> 1), p, rank, mb, nb);
    col0 = nb * TW + (v & 1) * (TW / 2);
    return TW / 2;
}

// Wait for phase `parity` of `bar`, giving up after `limit` ns or when another
// role has aborted.  A give-up by this wait records `site` in the status word.
static __device__ __noinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* status,
                                          uint64_t limit, int site) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > limit) {
            *abort_flag = 1;
            atomicCAS(status, 0, STATUS_TIMEOUT | site);
            __threadfence();
            return false;
        }
    }
}

// The same wait with its first polls inline, for the MMA issuer: it waits
// once per K chunk, and a call on that path showed up as idle tensor-pipe
// cycles.  After INLINE_POLLS failed polls it continues in wait_bounded, whose
// time limit then applies.
constexpr int INLINE_POLLS = 64;
__device__ __forceinline__ bool wait_fast(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* status,
                                          uint64_t limit, int site) {
#pragma unroll 1
    for (int i = 0; i < INLINE_POLLS; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return wait_bounded(bar, parity, abort_flag, status, limit, site);
}

// Bounded wait that ignores the abort flag: used to drain a role's own
// asynchronous work before the CTA exits.
static __device__ __noinline__ bool wait_drain(uint32_t bar, uint32_t parity, uint64_t limit) {
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit) return false;
    }
}

template <int OUT>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    if constexpr (OUT == SG_F16) {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    } else {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    }
}

template <int OUT>
__device__ __forceinline__ uint32_t pack2_relu(float lo, float hi) {
    if constexpr (OUT == SG_F16) {
        return cvt_relu_f16x2(lo, hi);
    } else {
        return cvt_relu_bf16x2(lo, hi);
    }
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// C without a TMA-legal layout: the warp's 32 x COLS block, already in its
// staging buffer in the TMA store's layout (row r at r * 128 bytes, 16-byte
// chunk j at chunk j ^ (r mod 8)), is written one row at a time, lane l
// taking columns l, l + 32, ...: each store instruction writes consecutive
// elements of one row.  Elements past M or N are not written.  Not inlined:
// the kernel's other paths keep the registers this fallback would take.
template <int OUT, int COLS>
static __device__ __noinline__ void store_rows(const Params& p, uint32_t buf, int row0, int col0, int lane) {
    constexpr int EB = (OUT == SG_F32) ? 4 : 2;  // output bytes per element
#pragma unroll 4
    for (int r = 0; r < 32; ++r) {
        const int row = row0 + r;
        if (row >= p.M) break;  // warp-uniform; the rows after it are past M too
#pragma unroll
        for (int h = 0; h < COLS / 32; ++h) {
            const int e = h * 32 + lane;
            const int col = col0 + e;
            if (col < p.N) {
                const uint32_t byte = static_cast<uint32_t>(e * EB);
                const uint32_t addr = buf + static_cast<uint32_t>(r) * 128u +
                                      (((byte >> 4) ^ static_cast<uint32_t>(r & 7)) << 4) + (byte & 15u);
                const int64_t idx = static_cast<int64_t>(row) * p.ldc + col;
                if constexpr (OUT == SG_F32) {
                    float x;
                    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(x) : "r"(addr));
                    static_cast<float*>(p.C)[idx] = x;
                } else {
                    unsigned short x;
                    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(x) : "r"(addr));
                    static_cast<unsigned short*>(p.C)[idx] = x;
                }
            }
        }
    }
}

template <int OUT>
__device__ __forceinline__ float load_one(const void* X, int64_t idx) {
    if constexpr (OUT == SG_F32) {
        return __ldg(static_cast<const float*>(X) + idx);
    } else if constexpr (OUT == SG_F16) {
        return __half2float(__ldg(static_cast<const __half*>(X) + idx));
    } else {
        return __bfloat162float(__ldg(static_cast<const __nv_bfloat16*>(X) + idx));
    }
}

// Adds this lane's row of a residual tile that TMA placed, 128-byte
// swizzled, in the staging buffer (row `lane` at lane * 128, 16-byte chunk j
// at j ^ (lane mod 8)) -- the same layout the store path writes.
template <int OUT, int COLS>
__device__ __forceinline__ void add_staged_residual(float (&v)[COLS], uint32_t rowaddr, int lane) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint32_t w[4];
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                     : "r"(rowaddr + ((j ^ (lane & 7)) << 4))
                     : "memory");
        if constexpr (OUT == SG_F32) {
#pragma unroll
            for (int t = 0; t < 4; ++t) v[4 * j + t] += __uint_as_float(w[t]);
        } else {
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                float lo, hi;
                if constexpr (OUT == SG_F16) {
                    const __half2 h = *reinterpret_cast<const __half2*>(&w[t]);
                    lo = __low2float(h);
                    hi = __high2float(h);
                } else {
                    const __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&w[t]);
                    lo = __low2float(h);
                    hi = __high2float(h);
                }
                v[8 * j + 2 * t] += lo;
                v[8 * j + 2 * t + 1] += hi;
            }
        }
    }
}

// Mode 5: one warp's share of decoding the integer-coded B into the
// resident panel.  The panel has the layout TMA gives a 16-bit B: K chunk
// kc and column block nb (of 128 columns) at (kc * n_blocks + nb) *
// block_bytes, 64-column box j of it at j * box_bytes, K row r of the box at
// r * 128 bytes, and its 16-byte chunk c (8 columns) at position c ^ (r mod
// 8) (the 128-byte swizzle).  A code becomes the 16-bit value equal to it
// (exact: |code| <= 128); codes past K or N are written as 0, the zero fill
// of a TMA load.  Warp `part` of `nparts` takes every nparts-th group of 32
// chunks.  The panel is decoded before any MMA can start, so each lane
// issues the loads of DEC_UNROLL chunks (8 codes each: one 8-byte load when
// the codes are 8-byte aligned) before it converts any of them.
constexpr int DEC_UNROLL = 16;
__device__ __forceinline__ void decode_panel(uint32_t panel, const Params& p, int n_blocks, int k_chunks,
                                             uint32_t block_bytes, uint32_t box_bytes, int part, int nparts,
                                             int lane) {
    const int chunks = n_blocks * 16;  // 16-byte chunks in one K row of the panel
    const int total = k_chunks * 64 * chunks;
    const int step = nparts * 32;
    const bool vec = ((reinterpret_cast<uintptr_t>(p.Bq) | static_cast<uintptr_t>(p.ldb)) & 7) == 0;
    for (int t0 = part * 32 + lane; t0 < total; t0 += step * DEC_UNROLL) {
        uint2 codes[DEC_UNROLL];
#pragma unroll
        for (int u = 0; u < DEC_UNROLL; ++u) {
            const int t = t0 + u * step;
            const int k = t / chunks, n0 = (t % chunks) * 8;
            codes[u] = make_uint2(0u, 0u);
            if (t < total && k < p.K && n0 < p.N) {
                const int8_t* src = p.Bq + static_cast<int64_t>(k) * p.ldb + n0;
                if (vec && n0 + 8 <= p.N) {
                    codes[u] = __ldg(reinterpret_cast<const uint2*>(src));
                } else {
                    uint32_t lo = 0, hi = 0;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint32_t byte = (n0 + i < p.N) ? static_cast<uint8_t>(__ldg(src + i)) : 0u;
                        if (i < 4) lo |= byte << (8 * i);
                        else hi |= byte << (8 * (i - 4));
                    }
                    codes[u] = make_uint2(lo, hi);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < DEC_UNROLL; ++u) {
            const int t = t0 + u * step;
            if (t >= total) break;
            const int k = t / chunks, n0 = (t % chunks) * 8;
            const int kc = k >> 6, r = k & 63, nb = n0 >> 7, col = n0 & 127;
            uint32_t w[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const uint32_t word = h < 2 ? codes[u].x : codes[u].y;
                const int sh = 16 * (h & 1);
                const float lo = static_cast<float>(static_cast<int8_t>((word >> sh) & 0xFFu));
                const float hi = static_cast<float>(static_cast<int8_t>((word >> (sh + 8)) & 0xFFu));
                if (p.in_bf16) {
                    __nv_bfloat162 x = __floats2bfloat162_rn(lo, hi);
                    w[h] = *reinterpret_cast<uint32_t*>(&x);
                } else {
                    __half2 x = __floats2half2_rn(lo, hi);
                    w[h] = *reinterpret_cast<uint32_t*>(&x);
                }
            }
            const uint32_t c = static_cast<uint32_t>((col & 63) >> 3);
            st_shared_v4(panel + static_cast<uint32_t>(kc * n_blocks + nb) * block_bytes + (col >> 6) * box_bytes +
                             r * 128 + ((c ^ static_cast<uint32_t>(r & 7)) << 4),
                         w[0], w[1], w[2], w[3]);
        }
    }
}

// Mode 5: v * scale[col] + bias[col] for the COLS columns starting at col0,
// one multiply-add per element (each rounded once; the tolerance covers
// it), with the scales at par + 4 * col and the biases (zeros without a
// bias) at par + nbias + 4 * col in shared memory, copied there once per
// CTA and zero past N.  Every lane reads the same addresses (broadcast).
template <int COLS>
__device__ __forceinline__ void scale_bias_smem(float (&v)[COLS], uint32_t par, uint32_t nbias, int col0) {
#pragma unroll
    for (int i = 0; i < COLS / 4; ++i) {
        const uint32_t off = static_cast<uint32_t>(col0 + 4 * i) * 4u;
        float s0, s1, s2, s3, b0, b1, b2, b3;
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(s0), "=f"(s1), "=f"(s2), "=f"(s3) : "r"(par + off));
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(b0), "=f"(b1), "=f"(b2), "=f"(b3)
                     : "r"(par + nbias + off));
        v[4 * i + 0] = fmaf(v[4 * i + 0], s0, b0);
        v[4 * i + 1] = fmaf(v[4 * i + 1], s1, b1);
        v[4 * i + 2] = fmaf(v[4 * i + 2], s2, b2);
        v[4 * i + 3] = fmaf(v[4 * i + 3], s3, b3);
    }
}

// + bias[col] for the COLS columns starting at col0, from the copy of the
// biases staged in shared memory at `par` (zero past N; col0 + COLS lies
// within the staged columns).
template <int COLS>
__device__ __forceinline__ void add_bias_smem(float (&v)[COLS], uint32_t par, int col0) {
#pragma unroll
    for (int i = 0; i < COLS / 4; ++i) {
        float b0, b1, b2, b3;
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(b0), "=f"(b1), "=f"(b2), "=f"(b3)
                     : "r"(par + static_cast<uint32_t>(col0 + 4 * i) * 4u));
        v[4 * i + 0] += b0;
        v[4 * i + 1] += b1;
        v[4 * i + 2] += b2;
        v[4 * i + 3] += b3;
    }
}

// + bias[col] for the COLS columns starting at col0 (zero past N).
template <int COLS>
__device__ __forceinline__ void add_bias(float (&v)[COLS], const float* __restrict__ bias, int col0, int N) {
    if (col0 + COLS <= N && (reinterpret_cast<uintptr_t>(bias + col0) & 15) == 0) {
        const float4* b4 = reinterpret_cast<const float4*>(bias + col0);
#pragma unroll
        for (int i = 0; i < COLS / 4; ++i) {
            const float4 b = __ldg(b4 + i);
            v[4 * i + 0] += b.x;
            v[4 * i + 1] += b.y;
            v[4 * i + 2] += b.z;
            v[4 * i + 3] += b.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < COLS; ++i) {
            const int col = col0 + i;
            v[i] += (col < N) ? __ldg(bias + col) : 0.0f;
        }
    }
}

// RES: the kernel adds a residual R (C = epilogue(A . B + R)); a separate
// instantiation, so the plain epilogue carries none of its work.  ESZ: the
// operands' element size, 2 (fp16 / bf16, kind::f16) or 1 (FP8 E4M3,
// kind::f8f6f4).
template <int BN, int OUT, int MODE, bool RES, int ESZ>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    sg_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmR,
                   const Params p) {
    static_assert(MODE == 1 || MODE == 3 || MODE == 4 || MODE == 5 || MODE == 6, "modes 1, 3, 4, 5 and 6");
    constexpr bool PANEL = (MODE == 4 || MODE == 5);      // B resident in shared memory
    constexpr bool DECODE = (MODE == 5);                  // ... decoded there from int8 codes
    static_assert(!DECODE || (ESZ == 2 && !RES), "mode 5: 16-bit A, no residual");
    constexpr bool WIDE = (MODE == 6);                    // two BN-wide accumulators per paired tile
    static_assert(!WIDE || BN == 256, "wide tiles hold two 256-column accumulators");
    constexpr bool PAIR = (MODE == 3 || WIDE);  // paired MMA (cta_group::2)
    constexpr int CM = PAIR ? 2 : 1;            // CTAs per cluster
    constexpr int NSUB = WIDE ? 2 : 1;          // accumulators per tile
    constexpr int TW = BN * NSUB;               // tile width in columns
    constexpr int CG = PAIR ? 2 : 1;            // cta_group of every tcgen05 instruction
    constexpr int BL = PAIR ? TW / 2 : BN;      // B columns staged by this CTA
    using L = Layout<BN, BL>;
    using G = Geom<ESZ>;
    static_assert(BL % G::BOXC == 0, "B is staged in whole 128-byte-wide boxes");
    constexpr uint16_t CLUSTER_MASK = static_cast<uint16_t>((1u << CM) - 1u);
    const uint32_t rank = (CM > 1) ? cluster_ctarank() : 0u;
    const int cluster_id = static_cast<int>(blockIdx.x) / CM;
    const int num_clusters = static_cast<int>(gridDim.x) / CM;
    constexpr int ACC = L::ACC;
    constexpr int COLS = (OUT == SG_F32) ? 32 : 64;  // output columns per 128-byte staging row
    static_assert(BN % COLS == 0, "tile width must hold whole staging rows");

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + SMEM_ALIGN - 1) & ~static_cast<uint32_t>(SMEM_ALIGN - 1);
    uint8_t* gbase = smem_raw + (base - raw);
    const int stages = p.stages;
    // slots per ring barrier pair; a group must divide the ring
    const int ring_group = (p.ring_group == 2 && stages % 2 == 0 && p.a_tma && p.b_tma) ? 2 : 1;
    // Shared-memory map.  Modes 1-3: [ring][staging][barriers].  Modes 4
    // and 5: [resident B: k_chunks x n_blocks blocks of BN columns][ring of A
    // tiles, each k_chunks A chunks][staging][mode 5: scales, biases; mode 4
    // with a bias: biases][barriers].
    constexpr int B_BLOCK_BYTES = (BN / G::BOXC) * G::B_BOX_BYTES;  // one K chunk of one column block
    const uint32_t res_bytes = PANEL ? static_cast<uint32_t>(p.k_chunks * p.n_blocks) * B_BLOCK_BYTES : 0u;
    const uint32_t stage_bytes = PANEL ? static_cast<uint32_t>(p.k_chunks) * A_STAGE_BYTES : L::STAGE_BYTES;
    const uint32_t ring0 = base + res_bytes;
    const uint32_t epi_off = res_bytes + static_cast<uint32_t>(stages) * stage_bytes;
    // mode 5: per-column scales then biases, fp32, n_blocks * BN of each
    const uint32_t par_nbias = DECODE ? static_cast<uint32_t>(p.n_blocks) * BN * 4u : 0u;
    // mode 4 with a bias: the biases alone, read from shared memory by every
    // tile (a bias read from global memory per chunk cost its whole latency)
    const bool bias_smem = PANEL && !DECODE && p.epi == SG_EPI_BIAS_RELU;
    const uint32_t par_bias = bias_smem ? static_cast<uint32_t>(p.n_blocks) * BN * 4u : 0u;
    const uint32_t par_off = epi_off + EPI_WARPS * EPI_BUF_BYTES;
    const uint32_t bar_off = par_off + 2u * par_nbias + par_bias;

    const uint32_t bar0 = base + bar_off;
    // barrier slots: full[0..7], empty[8..15], tmem_full[16..19], tmem_empty[20..23], drain[24],
    // then the tensor-memory address and abort flag, then residual[0..7] at 32..39
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (SG_MAX_STAGES + s); };
    auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * SG_MAX_STAGES + b); };
    auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * SG_MAX_STAGES + MAX_ACC + b); };
    const uint32_t drain_bar = bar0 + 8u * (2 * SG_MAX_STAGES + 2 * MAX_ACC);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + bar_off + 8 * (2 * SG_MAX_STAGES + 2 * MAX_ACC + 1));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    auto rres_bar = [&](int e) { return bar0 + 8u * (32 + e); };  // residual tile landed (one per epilogue warp)
    const uint32_t bres_bar = bar0 + 8u * 40;                      // mode 4: the resident B has landed

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < ACC; ++b) {
            mbar_init(tfull_bar(b), 1);
            mbar_init(tempty_bar(b), PAIR ? 2 * EPI_WARPS : EPI_WARPS);  // paired: both CTAs' epilogues
        }
        mbar_init(drain_bar, 1);
        for (int e = 0; e < EPI_WARPS; ++e) mbar_init(rres_bar(e), 1);
        mbar_init(bres_bar, DECODE ? EPI_WARPS : 1);  // mode 5: every epilogue warp decodes a share
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        if (p.k_chunks > 0) {
            if (p.a_tma) prefetch_tmap(&tmA);
            if (p.b_tma) prefetch_tmap(&tmB);
        }
        if (p.tma_store) prefetch_tmap(&tmC);
        if (RES && p.r_tma) prefetch_tmap(&tmR);
    }
    __syncwarp();  // reconverge before the warp-collective (.sync.aligned) instructions below
    if (warp == 1) {
        tmem_alloc<CG>(smem_addr(tmem_slot), TMEM_COLS);
        tmem_relinquish<CG>();
    }
    tc_fence_before();
    // the peer's barriers must be initialised before any copy or commit of the pair reaches them
    if constexpr (CM > 1) {
        cluster_sync();
    } else {
        __syncthreads();
    }
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0 && MODE == 1 && !(p.a_tma && p.b_tma)) {
        // ------------------------------------------------ element-load producer
        // (an operand without a TMA-legal layout; the whole warp copies)
        if (p.k_chunks > 0) {
            uint32_t slot = 0, phase = 0;
            uint32_t issued = 0, last_parity = 0;  // slots with TMA bytes in flight
            const uint32_t tx = (p.a_tma ? A_STAGE_BYTES : 0) + (p.b_tma ? L::B_STAGE_BYTES : 0);
            int64_t it = 0;
            bool ok = true;
            for (int tile = cluster_id; ok && tile < p.num_tiles; tile += num_clusters) {
                int mb, nb;
                tile_coords<CM>(tile, p, rank, mb, nb);
                for (int kc = 0; kc < p.k_chunks; ++kc, ++it) {
                    const bool w = wait_bounded(empty_bar(slot), phase ^ 1u, abort_flag, p.status, p.wait_limit_ns,
                                                SITE_PRODUCER_EMPTY);
                    if (!__all_sync(0xffffffffu, w)) {
                        ok = false;
                        break;
                    }
                    if (it != p.skip_load) {
                        const uint32_t sa = ring0 + slot * stage_bytes;
                        if (lane == 0 && tx > 0) {
                            mbar_expect_tx(full_bar(slot), tx);
                            if (p.a_tma) tma_load_2d(sa, &tmA, full_bar(slot), kc * G::KB, mb * BM);
                            if (p.b_tma) {
#pragma unroll
                                for (int j = 0; j < BN / G::BOXC; ++j)
                                    tma_load_2d(sa + A_STAGE_BYTES + j * G::B_BOX_BYTES, &tmB, full_bar(slot),
                                                nb * BN + j * G::BOXC, kc * G::KB);
                            }
                            issued |= 1u << slot;
                            last_parity = (last_parity & ~(1u << slot)) | (phase << slot);
                        }
                        if (!p.a_tma) copy_a_elements<ESZ>(sa, p, mb * BM, kc * G::KB, lane);
                        if (!p.b_tma) copy_b_elements<ESZ>(sa + A_STAGE_BYTES, p, kc * G::KB, nb * BN, BN, lane);
                        // the MMA reads these bytes through the async proxy
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(full_bar(slot));
                    }
                    if (++slot == static_cast<uint32_t>(stages)) {
                        slot = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok && lane == 0) {
                for (int s = 0; s < stages; ++s)
                    if ((issued >> s) & 1u) wait_drain(full_bar(s), (last_parity >> s) & 1u, p.wait_limit_ns);
            }
        }
    } else if (warp == 0) {
        // ------------------------------------------------ TMA producer
        // one elected thread issues every copy
        if (elect_one_sync() && p.k_chunks > 0) {
            uint32_t slot = 0, phase = 0;
            uint32_t issued = 0, last_parity = 0;  // per slot: ever filled, parity of its last fill
            int64_t it = 0;
            bool ok = true;
            if constexpr (PANEL && !DECODE) {
                // the resident B: every K chunk of every column block, once
                mbar_arrive_expect_tx(bres_bar, res_bytes);
                for (int kc = 0; kc < p.k_chunks; ++kc)
                    for (int nb = 0; nb < p.n_blocks; ++nb)
#pragma unroll
                        for (int j = 0; j < BN / G::BOXC; ++j)
                            tma_load_2d(base + (kc * p.n_blocks + nb) * B_BLOCK_BYTES + j * G::B_BOX_BYTES, &tmB,
                                        bres_bar, nb * BN + j * G::BOXC, kc * G::KB);
            }
            for (int tile = cluster_id; ok && tile < p.num_tiles; tile += num_clusters) {
                int mb = tile, col0 = 0, width = BN;
                if constexpr (!PANEL) width = unit_coords<CM, TW, ESZ>(tile, p, rank, mb, col0);
                // B columns landing in this CTA per K chunk: the paired MMA stages
                // half of the unit's columns in each CTA
                const int bl = PAIR ? width / 2 : width;
                const uint32_t chunk_tx = A_STAGE_BYTES + static_cast<uint32_t>(bl) * BK_BYTES;
                const int fills = PANEL ? 1 : p.k_chunks;  // mode 4: one ring slot holds every K chunk of A
                const int grp = PANEL ? 1 : ring_group;
                // paired: each accumulator's columns (sw of them) are split
                // between the two CTAs, this CTA staging [rank * sw / 2, +sw / 2)
                // of each in bps boxes
                const int sw = WIDE ? BN : width;
                const int bps = (sw / 2) / G::BOXC;
                for (int kc = 0; kc < fills; kc += grp, it += grp) {
                    if (!wait_bounded(empty_bar(slot), phase ^ 1u, abort_flag, p.status, p.wait_limit_ns,
                                      SITE_PRODUCER_EMPTY)) {
                        ok = false;
                        break;
                    }
                    const int nq = min(grp, fills - kc);  // K chunks in this group of slots
                    if (p.skip_load < it || p.skip_load >= it + nq) {
                        const uint32_t sa = ring0 + slot * stage_bytes;
                        if constexpr (PANEL) {
                            mbar_arrive_expect_tx(full_bar(slot), stage_bytes);
                            for (int c = 0; c < p.k_chunks; ++c)
                                tma_load_2d(sa + c * A_STAGE_BYTES, &tmA, full_bar(slot), c * G::KB, mb * BM);
                        } else if constexpr (PAIR) {
                            // both CTAs' copies complete on the even CTA's barrier
                            const uint32_t fb = mapa_shared(full_bar(slot), 0);
                            if (rank == 0) mbar_arrive_expect_tx(full_bar(slot), nq * 2 * chunk_tx);
                            for (int c = 0; c < nq; ++c) {
                                const uint32_t sc = sa + c * stage_bytes;
                                const int k0 = (kc + c) * G::KB;
                                tma_load_2d_pair(sc, &tmA, fb, k0, mb * BM);
                                for (int j = 0; j < bl / G::BOXC; ++j)
                                    tma_load_2d_pair(sc + A_STAGE_BYTES + j * G::B_BOX_BYTES, &tmB, fb,
                                                     col0 + (j / bps) * sw + static_cast<int>(rank) * (sw / 2) +
                                                         (j % bps) * G::BOXC,
                                                     k0);
                            }
                        } else {
                            mbar_arrive_expect_tx(full_bar(slot), nq * chunk_tx);
                            for (int c = 0; c < nq; ++c) {
                                const uint32_t sc = sa + c * stage_bytes;
                                const int k0 = (kc + c) * G::KB;
                                tma_load_2d(sc, &tmA, full_bar(slot), k0, mb * BM);
                                for (int j = 0; j < width / G::BOXC; ++j)
                                    tma_load_2d(sc + A_STAGE_BYTES + j * G::B_BOX_BYTES, &tmB, full_bar(slot),
                                                col0 + j * G::BOXC, k0);
                            }
                        }
                        issued |= 1u << slot;
                        last_parity = (last_parity & ~(1u << slot)) | (phase << slot);
                    }
                    slot += grp;
                    if (slot == static_cast<uint32_t>(stages)) {
                        slot = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok && (!PAIR || rank == 0)) {
                // the CTA is leaving early: let this warp's copies land first (paired: the
                // even CTA's barriers also count the odd CTA's copies)
                for (int s = 0; s < stages; ++s)
                    if ((issued >> s) & 1u) wait_drain(full_bar(s), (last_parity >> s) & 1u, p.wait_limit_ns);
                if (PANEL && !DECODE) wait_drain(bres_bar, 0, p.wait_limit_ns);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        // One elected thread runs the whole loop: its waits, its tcgen05
        // instructions and its commits (a commit covers the MMAs its own
        // thread issued).  Measured on GB300 against the whole warp running
        // the loop with one lane issuing: the same on 8192^3, 2% faster where
        // the MMAs are short (128-column tiles).
        if (p.k_chunks > 0 && (!PAIR || rank == 0) && elect_one_sync()) {
            constexpr bool issuer = true;
            auto wait_all = [&](uint32_t bar, uint32_t parity, int site) {
                return wait_fast(bar, parity, abort_flag, p.status, p.wait_limit_ns, site);
            };
            uint32_t slot = 0, phase = 0;
            uint32_t ab = 0, aph = 0;  // accumulator index and its phase
            bool ok = true;
            if constexpr (PANEL) {
                ok = wait_all(bres_bar, 0, SITE_MMA_FULL);
                if (ok) tc_fence_after();
            }
            for (int tile = cluster_id; ok && tile < p.num_tiles; tile += num_clusters) {
                if constexpr (PANEL) {
                    // one A slot, every column block of the resident B
                    if (!wait_all(full_bar(slot), phase, SITE_MMA_FULL)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = ring0 + slot * stage_bytes;
                    for (int nb = 0; nb < p.n_blocks; ++nb) {
                        if (!wait_all(tempty_bar(ab), aph ^ 1u, SITE_MMA_TMEM_EMPTY)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t d_tmem = tmem_base + ab * BN;
                        if (issuer) {
                            for (int kc = 0; kc < p.k_chunks; ++kc) {
                                const uint64_t a_desc = smem_desc_sw128(sa + kc * A_STAGE_BYTES, 16, 1024);
                                const uint64_t b_desc = smem_desc_sw128(
                                    base + (kc * p.n_blocks + nb) * B_BLOCK_BYTES, G::B_BOX_BYTES, 1024);
                                const int ksteps = min(G::KB / G::UK, (p.K - kc * G::KB + G::UK - 1) / G::UK);
#pragma unroll
                                for (int k = 0; k < G::KB / G::UK; ++k) {
                                    if (k < ksteps)
                                        umma<ESZ>(d_tmem, a_desc + ((k * 32) >> 4),
                                                  b_desc + ((k * G::B_KSTEP_BYTES) >> 4), p.idesc,
                                                  (kc | k) != 0 ? 1u : 0u);
                                }
                            }
                            umma_commit(tfull_bar(ab));
                        }
                        if (++ab == static_cast<uint32_t>(ACC)) {
                            ab = 0;
                            aph ^= 1u;
                        }
                    }
                    if (!ok) break;
                    if (issuer) umma_commit(empty_bar(slot));  // the A slot is free once every block has read it
                    if (++slot == static_cast<uint32_t>(stages)) {
                        slot = 0;
                        phase ^= 1u;
                    }
                    continue;
                }
                int umb, ucol;
                const int uw = unit_coords<CM, TW, ESZ>(tile, p, rank, umb, ucol);
                const int nsub = WIDE ? uw / BN : 1;  // accumulators this unit fills
                const uint32_t idesc = (WIDE || uw == BN) ? p.idesc : p.idesc_half;
                // the unit's accumulators in rotation order; the first is claimed
                // now, the others just before their first MMA
                uint32_t sab[NSUB] = {}, saph[NSUB] = {};
#pragma unroll
                for (int h = 0; h < NSUB; ++h) {
                    if (h < nsub) {
                        sab[h] = ab;
                        saph[h] = aph;
                        if (++ab == static_cast<uint32_t>(ACC)) {
                            ab = 0;
                            aph ^= 1u;
                        }
                    }
                }
                if (!wait_all(tempty_bar(sab[0]), saph[0] ^ 1u, SITE_MMA_TMEM_EMPTY)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // Slots come in groups of ring_group on one full and one empty
                // barrier: each wait stalls this warp long enough for the tensor
                // pipe to run dry, so fewer waits per MMA keep it busier.
                for (int kc = 0; kc < p.k_chunks; kc += ring_group) {
                    if (!wait_all(full_bar(slot), phase, SITE_MMA_FULL)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int nq = min(ring_group, p.k_chunks - kc);
#pragma unroll
                    for (int h = 0; h < NSUB; ++h) {
                        if (h >= nsub) break;
                        if (h > 0 && kc == 0) {
                            // a wide tile's next accumulator, claimed only now: the
                            // previous tile's epilogue drains it while the first
                            // accumulator's first MMAs run
                            if (!wait_all(tempty_bar(sab[h]), saph[h] ^ 1u, SITE_MMA_TMEM_EMPTY)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                        }
                        if (issuer) {
                            const uint32_t d_tmem = tmem_base + sab[h] * BN;
                            for (int c = 0; c < nq; ++c) {
                                const int kk = kc + c;
                                const uint32_t sa = ring0 + (slot + c) * stage_bytes;
                                // A: K-major, 8-row groups 1024 B apart.  B: MN-major, 8-K-row
                                // groups 1024 B apart, 64-column blocks one TMA box apart; a
                                // wide tile's second accumulator reads the boxes after the first's.
                                const uint64_t a_desc = smem_desc_sw128(sa, 16, 1024);
                                const uint64_t b_desc = smem_desc_sw128(
                                    sa + A_STAGE_BYTES + h * ((BN / 2) / G::BOXC) * G::B_BOX_BYTES, G::B_BOX_BYTES,
                                    1024);
                                // K steps that lie wholly past K would only add products of
                                // zero-filled elements: skip them
                                const int ksteps = min(G::KB / G::UK, (p.K - kk * G::KB + G::UK - 1) / G::UK);
#pragma unroll
                                for (int k = 0; k < G::KB / G::UK; ++k) {
                                    // K step of 16: +32 bytes along A's swizzled row, +2 groups of 8 rows of B
                                    if (k < ksteps) {
                                        const uint64_t ad = a_desc + ((k * 32) >> 4);  // +32 bytes of K along the row
                                        const uint64_t bd = b_desc + ((k * G::B_KSTEP_BYTES) >> 4);
                                        const uint32_t acc = (kk | k) != 0 ? 1u : 0u;
                                        if constexpr (PAIR) {
                                            umma_pair<ESZ>(d_tmem, ad, bd, idesc, acc);
                                        } else {
                                            umma<ESZ>(d_tmem, ad, bd, idesc, acc);
                                        }
                                    }
                                }
                            }
                            // A wide tile's earlier accumulators are complete once their
                            // last MMAs are: hand each to the epilogue before the next
                            // accumulator's last MMAs, so its reads overlap them and the
                            // next tile's first MMAs find it free.
                            if (WIDE && h + 1 < nsub && kc + ring_group >= p.k_chunks) {
                                umma_commit_pair_multicast(tfull_bar(sab[h]), CLUSTER_MASK);
                            }
                        }
                    }
                    if (!ok) break;
                    if (issuer) {
                        if constexpr (PAIR) {
                            umma_commit_pair_multicast(empty_bar(slot), CLUSTER_MASK);  // frees the slots in both CTAs
                        } else {
                            umma_commit(empty_bar(slot));
                        }
                    }
                    slot += ring_group;
                    if (slot == static_cast<uint32_t>(stages)) {
                        slot = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if (issuer) {
                    // the unit's last accumulator (a wide tile's earlier one was handed over above)
                    const uint32_t last = nsub > 1 ? sab[NSUB - 1] : sab[0];
                    if constexpr (PAIR) {
                        umma_commit_pair_multicast(tfull_bar(last), CLUSTER_MASK);  // both CTAs' epilogues
                    } else {
                        umma_commit(tfull_bar(last));
                    }
                }
            }
            // every MMA of this CTA has completed before tensor memory is released
            if (issuer) {
                if constexpr (PAIR) {
                    umma_commit_pair(drain_bar);
                } else {
                    umma_commit(drain_bar);
                }
            }
            wait_drain(drain_bar, 0, p.wait_limit_ns);
        }
    } else {
        // ------------------------------------------------ epilogue
        const int e = warp - 2;                   // 0 .. EPI_WARPS-1
        const int q = warp & 3;                   // the tensor-memory lane quarter this warp may read
        constexpr int SPLIT = EPI_WARPS / 4;      // warps sharing a quarter
        const int part = e / 4;                   // which of them: takes column chunks part, part+SPLIT, ...
        const uint32_t buf = base + epi_off + e * EPI_BUF_BYTES;
        // the lane that issues this warp's TMA copies and waits for them
        // (bulk groups belong to the thread that committed them)
        const bool leader = elect_one_sync();
        const bool r_staged = RES && p.r_tma;  // residual tiles arrive by TMA in the staging buffer
        uint32_t r_phase = 0;
        bool r_pending = false;                    // a residual load is in flight into `buf`
        // Starts the TMA load of the residual box this warp needs for output
        // columns col0.. (after the previous store has read the buffer).
        auto load_residual = [&](int row0, int col0) {
            if (leader) {
                bulk_wait_group_read<0>();
                mbar_arrive_expect_tx(rres_bar(e), EPI_BUF_BYTES);
                tma_load_2d(buf, &tmR, rres_bar(e), col0, row0);
            }
            r_pending = true;
        };
        if constexpr (DECODE) {
            // the panel is decoded once and read back by the MMAs of every row tile
            decode_panel(base, p, p.n_blocks, p.k_chunks, B_BLOCK_BYTES, G::B_BOX_BYTES, e, EPI_WARPS, lane);
            fence_proxy_async_smem();  // the MMA reads it through the async proxy
            __syncwarp();
            if (leader) mbar_arrive(bres_bar);
            // the per-column scales and biases, read by every chunk of every tile
            const bool has_bias = p.epi == SG_EPI_BIAS_RELU;
            for (int i = e * 32 + lane; i < p.n_blocks * BN; i += EPI_WARPS * 32) {
                const float sc = i < p.N ? __ldg(p.b_scale + i) : 0.0f;
                const float bi = (has_bias && i < p.N) ? __ldg(p.bias + i) : 0.0f;
                asm volatile("st.shared.f32 [%0], %1;" ::"r"(base + par_off + 4u * i), "f"(sc) : "memory");
                asm volatile("st.shared.f32 [%0], %1;" ::"r"(base + par_off + par_nbias + 4u * i), "f"(bi) : "memory");
            }
            // all eight epilogue warps have written their share before any reads it
            asm volatile("bar.sync 1, %0;" ::"r"(EPI_WARPS * 32) : "memory");
        }
        if (bias_smem) {
            // mode 4's biases (zero past N), read by every chunk of every tile
            for (int i = e * 32 + lane; i < p.n_blocks * BN; i += EPI_WARPS * 32) {
                const float bi = i < p.N ? __ldg(p.bias + i) : 0.0f;
                asm volatile("st.shared.f32 [%0], %1;" ::"r"(base + par_off + 4u * i), "f"(bi) : "memory");
            }
            asm volatile("bar.sync 1, %0;" ::"r"(EPI_WARPS * 32) : "memory");
        }
        uint32_t ab = 0, aph = 0;
        // accumulators: one per unit (modes 1, 3), one per column block of a row
        // tile (modes 4, 5), one per BN columns of a unit (mode 6)
        int subs = PANEL ? p.n_blocks : 1;
        for (int tile = cluster_id, sub = 0; tile < p.num_tiles;) {
            int mb = tile, ucol = sub * BN, width = BN;
            if constexpr (WIDE) {
                int u0;
                subs = unit_coords<CM, TW, ESZ>(tile, p, rank, mb, u0) / BN;
                ucol = u0 + sub * BN;
            } else if constexpr (!PANEL) {
                width = unit_coords<CM, TW, ESZ>(tile, p, rank, mb, ucol);
            }
            const int row0 = mb * BM + q * 32;
            const int row = row0 + lane;
            // the residual of this warp's first chunk loads while the MMAs run
            if (r_staged && row0 < p.M && ucol + part * COLS < p.N) load_residual(row0, ucol + part * COLS);
            if (p.k_chunks > 0) {
                const bool w = wait_bounded(tfull_bar(ab), aph, abort_flag, p.status, p.wait_limit_ns,
                                            SITE_EPI_TMEM_FULL);
                if (!__all_sync(0xffffffffu, w)) break;
                tc_fence_after();
            }
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + ab * BN;
            // Mode 6, 16-bit output, no residual: this warp's columns of the
            // accumulator are read into registers (converted and packed) and
            // the accumulator handed back before any of them is stored.  The
            // next tile's MMAs need this accumulator after a few of their first
            // MMAs, so the tile boundary waits only for the reads.
            constexpr bool EARLY = WIDE && OUT != SG_F32 && !RES;
            if (EARLY && p.k_chunks > 0 && p.tma_store) {
                constexpr int NCH = BN / (SPLIT * COLS);  // this warp's 64-column chunks
                uint32_t pk[NCH][COLS / 2];
                const bool relu = p.epi != SG_EPI_NONE;
#pragma unroll
                for (int i = 0; i < NCH; ++i) {
                    const int c = part * COLS + i * SPLIT * COLS;
                    uint32_t r[32], r2[32];
                    tmem_ld_32x32b_x32(t_row + c, r);
                    tmem_ld_32x32b_x32(t_row + c + 32, r2);
                    tmem_wait_ld_dep(r);
                    tmem_wait_ld_dep(r2);  // already complete; orders the uses of r2
                    float v[COLS];
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        v[j] = __uint_as_float(r[j]);
                        v[32 + j] = __uint_as_float(r2[j]);
                    }
                    if (p.epi == SG_EPI_BIAS_RELU) add_bias<COLS>(v, p.bias, ucol + c, p.N);
#pragma unroll
                    for (int j = 0; j < COLS / 2; ++j)
                        pk[i][j] = relu ? pack2_relu<OUT>(v[2 * j], v[2 * j + 1]) : pack2<OUT>(v[2 * j], v[2 * j + 1]);
                }
                // every value this warp needs is in registers: hand the accumulator back
                tc_fence_before();
                __syncwarp();
                if (leader) {
                    if constexpr (PAIR) {
                        mbar_arrive_cluster(mapa_shared(tempty_bar(ab), 0));
                    } else {
                        mbar_arrive(tempty_bar(ab));
                    }
                }
#pragma unroll
                for (int i = 0; i < NCH; ++i) {
                    const int col0 = ucol + part * COLS + i * SPLIT * COLS;
                    if (row0 < p.M && col0 < p.N) {  // warp-uniform: the box holds in-range elements
                        if (leader) bulk_wait_group_read<0>();  // the previous store has read the buffer
                        __syncwarp();
                        const uint32_t rowaddr = buf + lane * 128;
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            st_shared_v4(rowaddr + ((j ^ (lane & 7)) << 4), pk[i][4 * j], pk[i][4 * j + 1],
                                         pk[i][4 * j + 2], pk[i][4 * j + 3]);
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (leader) {
                            tma_store_2d(&tmC, buf, col0, row0);
                            bulk_commit_group();
                        }
                    }
                }
                __syncwarp();
                if (++ab == static_cast<uint32_t>(ACC)) {
                    ab = 0;
                    aph ^= 1u;
                }
                if (++sub == subs) {
                    sub = 0;
                    tile += num_clusters;
                }
                continue;
            }
#pragma unroll 1
            for (int c = part * COLS; c < width; c += SPLIT * COLS) {
                const int col0 = ucol + c;
                float v[COLS];
                if (p.k_chunks > 0) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(t_row + c, r);
                    if constexpr (COLS == 64) {
                        uint32_t r2[32];
                        tmem_ld_32x32b_x32(t_row + c + 32, r2);
                        tmem_wait_ld_dep(r);
                        tmem_wait_ld_dep(r2);  // already complete; orders the uses of r2
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[32 + i] = __uint_as_float(r2[i]);
                    } else {
                        tmem_wait_ld_dep(r);
                    }
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
                } else {
#pragma unroll
                    for (int i = 0; i < COLS; ++i) v[i] = 0.0f;
                }
                if constexpr (RES) {
                    if (r_staged) {
                        if (row0 < p.M && col0 < p.N) {  // warp-uniform: a residual box was loaded
                            const bool w = wait_bounded(rres_bar(e), r_phase, abort_flag, p.status, p.wait_limit_ns,
                                                        SITE_EPI_RESIDUAL);
                            if (!__all_sync(0xffffffffu, w)) break;
                            r_phase ^= 1u;
                            r_pending = false;
                            add_staged_residual<OUT, COLS>(v, buf + lane * 128, lane);
                        }
                    } else if (row < p.M) {
#pragma unroll
                        for (int i = 0; i < COLS; ++i) {
                            const int col = col0 + i;
                            if (col < p.N) v[i] += load_one<OUT>(p.R, static_cast<int64_t>(row) * p.ldr + col);
                        }
                    }
                }
                if constexpr (DECODE) {
                    scale_bias_smem<COLS>(v, base + par_off, par_nbias, col0);
                } else if (bias_smem) {
                    add_bias_smem<COLS>(v, base + par_off, col0);
                } else if (p.epi == SG_EPI_BIAS_RELU) {
                    add_bias<COLS>(v, p.bias, col0, p.N);
                }
                const bool relu = p.epi != SG_EPI_NONE;
                if (OUT == SG_F32 || !p.tma_store) {
                    if (relu) {
#pragma unroll
                        for (int i = 0; i < COLS; ++i) v[i] = (v[i] <= 0.0f) ? 0.0f : v[i];
                    }
                }
                if (p.tma_store) {
                    if (row0 < p.M && col0 < p.N) {  // warp-uniform: the box holds in-range elements
                        // the previous store has read the buffer (a staged residual already waited)
                        if (leader && !r_staged) bulk_wait_group_read<0>();
                        __syncwarp();
                        const uint32_t rowaddr = buf + lane * 128;
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            uint32_t w0, w1, w2, w3;
                            if constexpr (OUT == SG_F32) {
                                w0 = __float_as_uint(v[4 * j + 0]);
                                w1 = __float_as_uint(v[4 * j + 1]);
                                w2 = __float_as_uint(v[4 * j + 2]);
                                w3 = __float_as_uint(v[4 * j + 3]);
                            } else if (relu) {
                                w0 = pack2_relu<OUT>(v[8 * j + 0], v[8 * j + 1]);
                                w1 = pack2_relu<OUT>(v[8 * j + 2], v[8 * j + 3]);
                                w2 = pack2_relu<OUT>(v[8 * j + 4], v[8 * j + 5]);
                                w3 = pack2_relu<OUT>(v[8 * j + 6], v[8 * j + 7]);
                            } else {
                                w0 = pack2<OUT>(v[8 * j + 0], v[8 * j + 1]);
                                w1 = pack2<OUT>(v[8 * j + 2], v[8 * j + 3]);
                                w2 = pack2<OUT>(v[8 * j + 4], v[8 * j + 5]);
                                w3 = pack2<OUT>(v[8 * j + 6], v[8 * j + 7]);
                            }
                            // 128-byte swizzle: 16-byte chunk j of row r sits at chunk j ^ (r mod 8)
                            st_shared_v4(rowaddr + ((j ^ (lane & 7)) << 4), w0, w1, w2, w3);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (leader) {
                            tma_store_2d(&tmC, buf, col0, row0);
                            bulk_commit_group();
                        }
                    }
                } else if (row0 < p.M && col0 < p.N) {  // warp-uniform
                    // C without a TMA-legal layout: the block goes through the
                    // staging buffer in the same layout (the ReLU is already
                    // applied), then out row by row
                    const uint32_t rowaddr = buf + lane * 128;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        uint32_t w[4];
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            if constexpr (OUT == SG_F32) {
                                w[t] = __float_as_uint(v[4 * j + t]);
                            } else {
                                w[t] = pack2<OUT>(v[8 * j + 2 * t], v[8 * j + 2 * t + 1]);
                            }
                        }
                        st_shared_v4(rowaddr + ((j ^ (lane & 7)) << 4), w[0], w[1], w[2], w[3]);
                    }
                    __syncwarp();
                    store_rows<OUT, COLS>(p, buf, row0, col0, lane);
                }
                __syncwarp();  // the next tcgen05.ld is warp-collective; the buffer has been read
                // the next chunk's residual (the store just issued must read the buffer first)
                const int cn = c + SPLIT * COLS;
                if (r_staged && cn < width && row0 < p.M && ucol + cn < p.N) load_residual(row0, ucol + cn);
            }
            if (p.k_chunks > 0) {
                tc_fence_before();
                __syncwarp();
                if (leader) {
                    if constexpr (PAIR) {
                        mbar_arrive_cluster(mapa_shared(tempty_bar(ab), 0));  // the even CTA's MMA waits on it
                    } else {
                        mbar_arrive(tempty_bar(ab));
                    }
                }
            }
            if (++ab == static_cast<uint32_t>(ACC)) {
                ab = 0;
                aph ^= 1u;
            }
            if (++sub == subs) {
                sub = 0;
                tile += num_clusters;
            }
        }
        // leaving early with a residual load in flight: let it land first
        if (r_pending && leader) wait_drain(rres_bar(e), r_phase, p.wait_limit_ns);
        if (leader) bulk_wait_group<0>();
        __syncwarp();
    }

    __syncwarp();  // lanes that skipped a lane-0 role wait for it here
    tc_fence_before();
    // no CTA leaves while its peer may still copy into it or arrive on it
    if constexpr (CM > 1) {
        cluster_sync();
    } else {
        __syncthreads();
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<CG>(tmem_base, TMEM_COLS);
    }
}

}  // namespace sg
