// Tensor-core GEMMs of the ternary linear layer on sm_103a (tcgen05 + TMEM + TMA).
//
// Page "train_gpu.cu" (RWKV-x SR4 training driver): W_eff[r,c] = scale[c] *
// ternary(q)[r,c] (header comment "Optimizer split"); the backward products
// gq = grad*scale[c] and sgrad[c] = sum_r grad[r,c]*tern[r,c] (device glue
// kernels tg_gq, tg_scale_grad) with grad = X^T * dY.  The pages run these as a
// cuBLAS fp32 GEMM on a materialised W_eff followed by separate rows x cols
// passes; here each is one persistent tensor-core kernel:
//
//   forward : Y[m][c]  = scale[c] * (X * T)[m][c]        scale in the epilogue
//   dX      : dX[m][r] = (dY * W_hi^T + dY * W_lo^T)[m][r]  two MMAs per k-step
//                        into one TMEM accumulator; W_hi/W_lo = bf16 split of
//                        scale[c]*T, exact to 2^-17 relative
//   dW      : G = X^T * dY kept in TMEM; the epilogue writes gq = G*scale[c] and
//             reduces sum_r G*T per column from the 2-bit tiles (no stored G)
//
// GEMM convention inside a kernel: D[Mg][Ng] = sum_k A[m][k] * B[n][k], A and
// B bf16 in shared memory, D fp32 in TMEM.  A/B are "K-major" (k contiguous in
// global memory) or "MN-major" (m or n contiguous); both are read by TMA with
// the 128-byte (or 64-byte) swizzle that the tcgen05 shared-memory descriptors
// describe, so no operand is ever transposed in memory.
//
// Kernel shape: persistent, one CTA per SM; outputs of more than 128 rows use CTA
// pairs (a 2-CTA cluster, cta_group::2) on 256 x BN tiles, smaller ones single
// CTAs on 128 x BN tiles.  A launch walks the work units of a group of up to 8
// independent problems (one layer is a group of one).
//   warp 0     TMA producer (one thread): STAGES-deep ring of operand stages
//   warp 1     TMEM allocator + MMA issuer (one thread, the pair's leader)
//   warps 2-9  epilogue: TMEM -> registers -> global, two warps per TMEM lane quarter,
//              each taking half of a tile's columns (the 2-bit forward: warps 2-5, one per
//              quarter, and warps 6-13 expand the 2-bit T codes into bf16 operand tiles)
// Two TMEM accumulators (2 x BN columns) let the epilogue of tile i overlap the
// main loop of tile i+1.  Before exit the producer waits for the release of every
// stage it filled and the MMA thread for the release of the last accumulators, so
// no asynchronous arrival lands in shared memory the next kernel's CTA owns.
//
// Every mbarrier wait of the pipeline is bounded; on expiry a kernel records
// TERN_ERR_TIMEOUT in g_gemm_status (and the site in g_gemm_site), raises a CTA-wide
// abort flag, waits (again bounded) for its own TMA copies and MMAs in flight, frees
// TMEM and returns.  Three waits of the set-up have no bound, because the hardware
// offers none: the TMEM allocation (tcgen05.alloc blocks until the columns are
// free), the cluster barrier of a CTA pair (barrier.cluster) and the dependent-launch
// wait (griddepcontrol.wait).  The GEMMs are launched without programmatic stream
// serialization, so each one starts only after every earlier kernel on its stream has
// completed: no GEMM CTA shares an SM with a CTA that still holds TMEM, and its set-up
// never waits on another grid.
#include <algorithm>
#include <chrono>
#include <cmath>
#include <cstring>
#include <mutex>
#include <thread>
#include <type_traits>
#include <vector>

#include <cuda_bf16.h>

#include "common.cuh"

namespace tern {

__device__ int g_gemm_status;
// Failure diagnostics: GEMM CTAs counted at entry, after their set-up (TMEM
// allocation, cluster barrier, dependent-launch wait) and at exit, and where the
// first bounded wait gave up (site code, CTA, barrier's shared-memory address, parity).
__device__ unsigned long long g_gemm_count[3];   // CTAs entered, past set-up, exited
__device__ int g_gemm_site[4];

namespace {

constexpr int kBM = 128;           // rows of A (and of D) per CTA
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s per wait; a healthy wait takes microseconds

enum { EPI_FWD = 0, EPI_DX = 1, EPI_DW = 2 };
enum { SW128 = 2, SW64 = 4 };   // tcgen05 descriptor layout codes

struct GemmArgs {
    int Mg, Ng, Kg;
    int tiles_m, tiles_n, num_tiles, num_kb;
    float* out;               // [Mg][Ng] fp32 (Y, dX or gq); may be null for EPI_DW
    const float* scale;       // [Ng] column scale (EPI_FWD, EPI_DW)
    const uint32_t* packed;   // [Mg][Ng/16] 2-bit ternary codes (EPI_DW)
    float* partial;           // [ceil(Mg/128)*4][Ng] per-lane-quarter sgrad partials (EPI_DW)
    int accumulate;           // EPI_DW: gq += G*scale instead of gq = G*scale
    // Work units of this launch: unit u is tile tile_begin + u / split, k-blocks
    // [(u % split) * kb_per, ...).  With split > 1 (EPI_DW only) each unit writes
    // its raw partial tile to partial_g[u] and tern_dw_split_reduce finishes it.
    int tile_begin, num_units, split, kb_per;
    float* partial_g;
    uint16_t* out_bf16;       // [Mg][Ng] bf16 (RNE) copy of out, or its only output (EPI_FWD, EPI_DX)
    const uint32_t* bpacked;  // forward from 2-bit codes: T as [Kg][Ng/16] words (the B operand)
    const int* row_exp;       // dX from the fp16 + e4m3 split: dX row m is 2^row_exp[m] times the accumulator
};

// Up to G independent problems in one launch: their work units are concatenated
// (problem p owns units [unit_begin[p], unit_begin[p+1])) and each carries its
// own tensor maps and arguments.  A single problem is a group of one.
template <int G>
struct GemmGroup {
    CUtensorMap mA[G];
    CUtensorMap mB0[G];
    CUtensorMap mB1[G];
    GemmArgs args[G];
    int unit_begin[G + 1];
    int count;
};

// Problems per grouped launch: with three tensor maps each the parameter block stays under 4 KB.
constexpr int kGroup = 8;
static_assert(sizeof(GemmGroup<kGroup>) <= 4096, "kernel parameter block over 4 KB");

// The dX GEMM from the fp16 + e4m3 split reads four operands: A = dY16 (mA), B = h*T
// (mB0), A8 = dY8 (mA1), B8 = l*T (mB1).
template <int G>
struct GemmGroup4 {
    CUtensorMap mA[G];
    CUtensorMap mB0[G];
    CUtensorMap mB1[G];
    CUtensorMap mA1[G];
    GemmArgs args[G];
    int unit_begin[G + 1];
    int count;
};

template <class GRP>
__device__ __forceinline__ int group_find(const GRP& g, int unit) {
    int p = 0;
    while (p + 1 < g.count && unit >= g.unit_begin[p + 1]) ++p;
    return p;
}

// CG CTAs (1, or a 2-CTA cluster) share one MMA of M = 128*CG rows by N = BN columns.
// Each CTA loads its 128 rows of A and BN/CG rows of B per k-block of BK, and its
// TMEM holds its own 128 rows of D.
// PK: the B operand (the forward's T) is read as 2-bit codes and expanded to bf16 in
// shared memory by converter warps (warps 6-13: two teams of four that take alternate
// k-blocks) instead of being copied by TMA.
// F8: the dX GEMM from the fp16 + e4m3 split: per k-block a binary16 A and B (rows of
// BK*2 bytes, SW128) and an e4m3 A and B (rows of BK bytes, SW64), in that order.
template <int CG_, int BN_, int BK_, bool A_MN_, bool B_MN_, int NB_, int EPI_, int STAGES_, bool PK_ = false,
          bool F8_ = false>
struct Cfg {
    static constexpr int CG = CG_, BN = BN_, BK = BK_, NB = NB_, EPI = EPI_, STAGES = STAGES_;
    static constexpr bool A_MN = A_MN_, B_MN = B_MN_, PK = PK_, F8 = F8_;
    // warps: producer, MMA, EPI_WARPS epilogue warps (two per TMEM lane quarter, each taking
    // half the columns; four when PK), and for PK two teams of four converter warps
    static constexpr int EPI_WARPS = PK ? 4 : 8;
    static constexpr int THREADS = 64 + 32 * EPI_WARPS + (PK ? 256 : 0);
    static constexpr int TILE_M = kBM * CG;
    static constexpr int B_ROWS = BN / CG;
    static constexpr int A_BYTES = kBM * BK * 2;
    static constexpr int B_BYTES = B_ROWS * BK * 2;
    static constexpr int A8_BYTES = F8 ? kBM * BK : 0;
    static constexpr int B8_BYTES = F8 ? B_ROWS * BK : 0;
    static constexpr int STAGE_BYTES = A_BYTES + NB * B_BYTES + A8_BYTES + B8_BYTES;   // per CTA
    static constexpr int TX_BYTES = CG * (PK ? A_BYTES : STAGE_BYTES);   // TMA bytes on the leader's barrier
    static constexpr int P_BYTES = PK ? BK * (B_ROWS / 16) * 4 : 0;     // 2-bit codes of a stage's B (PK)
    // raster: runs of RASTER m-tiles share an n-tile (tile_coords).  dX's B operands (W_hi
    // and W_lo, or the split planes) are the larger panels, so its runs are longer.
    static constexpr int RASTER = (EPI == EPI_DX ? 24 : 16) / CG;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr int SMEM_BYTES = STAGES * (STAGE_BYTES + P_BYTES) + 1024 + 256;
    static_assert(CG == 1 || CG == 2, "CTA group");
    static_assert(BK == 64 || (BK == 32 && !A_MN && !B_MN), "MN-major operands use 64-deep k-blocks");
    static_assert(BN % 64 == 0 && BN <= 256 && B_ROWS % 64 == 0, "BN");
    static_assert(TMEM_COLS == 256 || TMEM_COLS == 512, "TMEM allocation must be a power of two");
    static_assert(SMEM_BYTES <= 232448, "shared memory");
    static_assert(!PK || (EPI == EPI_FWD && B_MN && NB == 1 && BK == 64) || (EPI == EPI_DX && !B_MN && NB == 2 && BK == 64),
                  "packed operand: the forward's T or dX's W_hi / W_lo");
    static_assert(!F8 || (EPI == EPI_DX && !A_MN && !B_MN && NB == 1 && BK == 64 && !PK), "fp16 + e4m3 split: dX");
};

// One CTA per 128 x 256 tile (small problems).
using Fwd1 = Cfg<1, 256, 64, false, true, 1, EPI_FWD, 4>;   // A = X (K-major), B = T [K][N] (MN-major)
using Dx1 = Cfg<1, 256, 32, false, false, 2, EPI_DX, 5>;    // A = dY (K-major), B = W_hi, W_lo (K-major)
using Dw1 = Cfg<1, 256, 64, true, true, 1, EPI_DW, 4>;      // A = X^T, B = dY^T (both MN-major)
// A CTA pair per 256 x 256 tile: half the shared-memory operand traffic per MMA.
using Fwd2 = Cfg<2, 256, 64, false, true, 1, EPI_FWD, 7>;
using Dx2 = Cfg<2, 256, 64, false, false, 2, EPI_DX, 4>;
using Dw2 = Cfg<2, 256, 64, true, true, 1, EPI_DW, 7>;
// The forward with T read as 2-bit codes.
using FwdP1 = Cfg<1, 256, 64, false, true, 1, EPI_FWD, 4, true>;
using FwdP2 = Cfg<2, 256, 64, false, true, 1, EPI_FWD, 6, true>;
// dX with W_hi and W_lo expanded from the 2-bit codes and a per-column s_hi / s_lo table.
using DxP1 = Cfg<1, 256, 64, false, false, 2, EPI_DX, 2, true>;
using DxP2 = Cfg<2, 256, 64, false, false, 2, EPI_DX, 4, true>;
// dX from the fp16 + e4m3 split.
using Dx8_1 = Cfg<1, 256, 64, false, false, 1, EPI_DX, 3, false, true>;
using Dx8_2 = Cfg<2, 256, 64, false, false, 1, EPI_DX, 4, false, true>;

// tcgen05 instruction descriptor: fp32 D, M x N, operand majors and the A/B format code
// (kind::f16: 0 = f16, 1 = bf16; kind::f8f6f4: 0 = e4m3).
__host__ __device__ constexpr uint32_t make_idesc(int M, int N, bool a_mn, bool b_mn, uint32_t fmt = 1u) {
    return (1u << 4)                       // D format: f32
           | (fmt << 7)                    // A format
           | (fmt << 10)                   // B format
           | (static_cast<uint32_t>(a_mn) << 15)
           | (static_cast<uint32_t>(b_mn) << 16)
           | (static_cast<uint32_t>(N >> 3) << 17)
           | (static_cast<uint32_t>(M >> 4) << 24);
}

// tcgen05 shared-memory matrix descriptor.
__device__ __forceinline__ uint64_t make_sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
    return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) |
           (static_cast<uint64_t>(layout) << 61);
}

// Descriptor of the kk-th 16-deep k-slice of an operand tile at `base`.
//  K-major, BK = 64: rows of 128 B (SW128), 8-row atoms 1024 B apart; the slice
//                    starts 32 B further along the row.
//  K-major, BK = 32: rows of 64 B (SW64), 8-row atoms 512 B apart.
//  MN-major (BK 64): 64-element MN chunks of BK k-rows (128 B each, SW128);
//                    chunks LBO = 64*BK*2 B apart, 8-k-row groups SBO = 1024 B
//                    apart; the slice starts two groups (2048 B) further.
template <bool MN, int BK>
__device__ __forceinline__ uint64_t op_desc(uint32_t base, int kk) {
    if constexpr (MN) {
        return make_sdesc(base + kk * 2048u, 64u * BK * 2u, 1024u, SW128);
    } else if constexpr (BK == 64) {
        return make_sdesc(base + kk * 32u, 16u, 1024u, SW128);
    } else {
        return make_sdesc(base + kk * 32u, 16u, 512u, SW64);
    }
}

// Grouped raster: runs of GM m-tiles share an n-tile, so neighbouring CTAs reuse
// the same B panel and A panels stay resident in L2.
template <int GM>
__host__ __device__ __forceinline__ void tile_coords(int tile, int tiles_m, int tiles_n, int& mt, int& nt) {
    const int group = tile / (GM * tiles_n);
    const int first_m = group * GM;
    const int gm = min(GM, tiles_m - first_m);
    const int local = tile - group * GM * tiles_n;
    mt = first_m + local % gm;
    nt = local / gm;
}

// Bounded wait on an mbarrier phase.  Returns false on timeout (after recording
// it) or, when `watch_abort`, once another role has raised the abort flag.
// Site codes: (epilogue kind + 1) * 100 + CTA group * 10 + role, role 1 producer
// stage wait, 2 producer tail, 3 MMA accumulator wait, 4 MMA stage wait, 5 MMA
// drain, 6 MMA tail, 7 epilogue accumulator wait, 8 copies after an abort; 999
// the self-test.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                             bool watch_abort, int site, uint64_t limit_ns = kWaitLimitNs) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    // The time waited is the sum of the timer's forward steps between polls, each
    // counted up to 1 ms: a timer that steps backwards, or jumps forward once, cannot
    // end a healthy wait.  A poll count backs the bound should the timer stall.
    uint64_t last = ptx::globaltimer(), waited = 0;
    for (uint32_t it = 1;; ++it) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (watch_abort && *abort_flag) return false;
            const uint64_t now = ptx::globaltimer();
            const int64_t step = static_cast<int64_t>(now - last);
            last = now;
            if (step > 0) waited += static_cast<uint64_t>(step < 1000000 ? step : 1000000);
            if (waited > limit_ns || it >= (1u << 30)) {
                *abort_flag = 1;
                atomicExch(&g_gemm_status, 1);
                if (atomicCAS(&g_gemm_site[0], 0, site) == 0) {
                    g_gemm_site[1] = static_cast<int>(blockIdx.x);
                    g_gemm_site[2] = static_cast<int>(bar);
                    g_gemm_site[3] = static_cast<int>(parity);
                }
                return false;
            }
        }
    }
}

// Sum over the 32 lanes of v[0..31] (lane l's row of a 32 x 32 block); on
// return lane l's v[0] holds the sum of column l.  Recursive halving, 31
// shuffles, fixed order.
__device__ __forceinline__ float warp_column_sums(float (&v)[32], int lane) {
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) {
        const bool upper = (lane & s) != 0;
#pragma unroll
        for (int i = 0; i < s; ++i) {
            const float send = upper ? v[i] : v[i + s];
            const float keep = upper ? v[i + s] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, s);
        }
    }
    return v[0];
}

// Store one 32 x 32 fp32 chunk of a warp (lane = row, v = its 32 columns) to global
// memory at `base` (row stride ld), rows < rows and columns < cols only.  Within each
// group of eight lanes the 8 x 8 block of 16-byte units is transposed by three butterfly
// stages of warp shuffles (no shared memory, which the operand pipeline keeps busy):
// afterwards lane l holds unit l & 7 of the group's eight rows, and each of the eight
// store instructions writes four whole 128-byte rows.  With add, the stored values are
// added to what is in memory (gradient accumulation).
__device__ __forceinline__ void store_chunk(float* base, int64_t ld, int rows, int cols, const float (&v)[32], bool add,
                                            int lane) {
    float4 u[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) u[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
#pragma unroll
    for (int d = 4; d >= 1; d >>= 1) {
        const bool upper = (lane & d) != 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (i & d) continue;
            const float4 send = upper ? u[i] : u[i | d];
            float4 recv;
            recv.x = __shfl_xor_sync(0xffffffffu, send.x, d);
            recv.y = __shfl_xor_sync(0xffffffffu, send.y, d);
            recv.z = __shfl_xor_sync(0xffffffffu, send.z, d);
            recv.w = __shfl_xor_sync(0xffffffffu, send.w, d);
            if (upper) u[i] = recv;
            else u[i | d] = recv;
        }
    }
    const int cq = lane & 7;   // this lane's 16-byte column group
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = (lane & ~7) + i;
        if (r < rows && 4 * cq < cols) {
            float4 x = u[i];
            float4* g = reinterpret_cast<float4*>(base + static_cast<int64_t>(r) * ld + 4 * cq);
            if (add) {
                const float4 o = *g;
                x = make_float4(o.x + x.x, o.y + x.y, o.z + x.z, o.w + x.w);
            }
            *g = x;
        }
    }
}

// Two weights of a packed word as one bf16 pair: t holds code i at bits 0-1 and code
// i+8 at bits 16-17 (the word shifted right by 2i); bit 0 of a code is "non-zero", bit 1
// "negative" (00 -> 0x0000, 01 -> 0x3F80 = +1, 11 -> 0xBF80 = -1).
__device__ __forceinline__ uint32_t tern_pair_bf16(uint32_t t) {
    return (t & 0x00010001u) * 0x3F80u | ((t << 14) & 0x80008000u);
}

// A tile's column scales, spread over the warp: lane l holds columns 8l..8l+7 of the
// tile starting at column col0 (zeros past the last column).  Loaded one tile ahead of
// their use, so that no chunk waits on a cold load.
__device__ __forceinline__ void load_tile_scales(const float* scale, int col0, int Ng, int lane, float (&sc)[8]) {
    const int c = col0 + 8 * lane;   // N % 16 == 0: the eight columns are all in range or all out
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
    if (scale != nullptr && c < Ng) {
        a = __ldg(reinterpret_cast<const float4*>(scale + c));
        b = __ldg(reinterpret_cast<const float4*>(scale + c + 4));
    }
    sc[0] = a.x, sc[1] = a.y, sc[2] = a.z, sc[3] = a.w, sc[4] = b.x, sc[5] = b.y, sc[6] = b.z, sc[7] = b.w;
}

// One 32-column chunk j of a warp's 32 rows: r[] is row `row` (the warp's rows start at
// `wrow`), columns c0..c0+31 (c0 = the tile's first column + 32j); sc holds the tile's
// scales as load_tile_scales spreads them.  tile128 is the index of the 128-row block
// the rows lie in.
template <class C>
__device__ __forceinline__ void epilogue_chunk(const GemmArgs& a, const uint32_t (&r)[32],
                                               const float (&sc)[8], int j, int row, int wrow, int c0, int tile128,
                                               int quad, int lane, int rexp = 0) {
    const bool row_ok = row < a.Mg;
    const bool hi_ok = c0 + 16 < a.Ng;   // N is a multiple of 16: the chunk's second half may lie past it
    float v[32];
    if constexpr (C::PK && C::EPI == EPI_FWD) {
        // the converters store columns i and i+8 of each 16-column group as the bf16 pair at
        // positions 2i, 2i+1: accumulator column 2i holds column i, 2i+1 holds i+8
#pragma unroll
        for (int g = 0; g < 2; ++g)
#pragma unroll
            for (int n = 0; n < 16; ++n) v[16 * g + n] = __uint_as_float(r[16 * g + 2 * (n & 7) + (n >> 3)]);
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
    }
    if constexpr (C::F8) {   // the dY row's exponent, taken out by the split
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = ldexpf(v[i], rexp);
    }
    if (C::EPI == EPI_FWD || (C::EPI == EPI_DW && a.out != nullptr)) {
        // column c0 + i of the chunk is register i % 8 of lane 4j + i / 8
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] *= __shfl_sync(0xffffffffu, sc[i & 7], 4 * j + (i >> 3));
    }
    // fp32 output (gq += ... with accumulate); the condition is the same for the whole warp
    if (a.out != nullptr && wrow < a.Mg)
        store_chunk(a.out + static_cast<int64_t>(wrow) * a.Ng + c0, a.Ng, a.Mg - wrow, a.Ng - c0, v,
                    C::EPI == EPI_DW && a.accumulate != 0, lane);
    if constexpr (C::EPI != EPI_DW) {
        if (a.out_bf16 != nullptr && row_ok) {   // 16 columns -> 32 bytes, round to nearest even
            const int64_t at = static_cast<int64_t>(row) * a.Ng + c0;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if (h == 0 || hi_ok) {
                    uint32_t b[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const __nv_bfloat162 t = __floats2bfloat162_rn(v[16 * h + 2 * q], v[16 * h + 2 * q + 1]);
                        b[q] = *reinterpret_cast<const uint32_t*>(&t);
                    }
                    uint4* ob = reinterpret_cast<uint4*>(a.out_bf16 + at + 16 * h);
                    ob[0] = make_uint4(b[0], b[1], b[2], b[3]);
                    ob[1] = make_uint4(b[4], b[5], b[6], b[7]);
                }
            }
        }
    }
    if constexpr (C::EPI == EPI_DW) {
        if (a.partial == nullptr) return;   // gq only
        // sgrad partial over this warp's 32 rows: sum_r G[r][c] * T[r][c]
        uint32_t w0 = 0, w1 = 0;
        if (row_ok) {
            const uint32_t* pr = a.packed + static_cast<int64_t>(row) * (a.Ng / 16) + c0 / 16;
            w0 = __ldg(pr);
            if (hi_ok) w1 = __ldg(pr + 1);
        }
        float t[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const uint32_t code = ((i < 16 ? w0 : w1) >> (2 * (i & 15))) & 3u;
            const float g = __uint_as_float(r[i]);
            t[i] = (code & 1u) ? ((code & 2u) ? -g : g) : 0.0f;
        }
        const float colsum = warp_column_sums(t, lane);
        if (c0 + lane < a.Ng) a.partial[static_cast<int64_t>(tile128 * 4 + quad) * a.Ng + c0 + lane] = colsum;
    }
}

template <class C, class GRP>
__device__ __forceinline__ void gemm_body(const GRP& grp) {
    constexpr int CG = C::CG;
    constexpr int SITE = (C::EPI + 1) * 100 + CG * 10;
    const int total_units = grp.unit_begin[grp.count];
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + C::STAGES * (C::STAGE_BYTES + C::P_BYTES));
    const uint32_t pring0 = base + static_cast<uint32_t>(C::STAGES * C::STAGE_BYTES);   // PK: codes of each stage
    // FULL, EMPTY (per stage), TFULL, TEMPTY (per accumulator), DRAIN, then (PK only) BREADY
    // (per stage: converters done with its B operand) and PFULL (per stage: its codes landed
    // in this CTA), then the TMEM address and abort flag
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * C::STAGES + 5 + (C::PK ? 2 * C::STAGES : 0));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const uint32_t bar0 = ptx::smem_u32(bars);
    const uint32_t FULL0 = bar0, EMPTY0 = bar0 + 8u * C::STAGES;
    const uint32_t TFULL0 = bar0 + 16u * C::STAGES, TEMPTY0 = TFULL0 + 16u, DRAIN = TFULL0 + 32u;
    const uint32_t BREADY0 = DRAIN + 8u, PFULL0 = BREADY0 + 8u * C::STAGES;

    if (threadIdx.x == 32) atomicAdd(&g_gemm_count[0], 1ull);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = CG == 2 ? ptx::cluster_ctarank() : 0u;   // 0 = leader of the pair
    const int unit = CG == 2 ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
    const int units = CG == 2 ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            ptx::mbar_init(FULL0 + 8u * s, 1);
            ptx::mbar_init(EMPTY0 + 8u * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(TFULL0 + 8u * b, 1);
            ptx::mbar_init(TEMPTY0 + 8u * b, C::EPI_WARPS * CG);   // every epilogue warp of the group
        }
        ptx::mbar_init(DRAIN, 1);
        if constexpr (C::PK) {
            for (int s = 0; s < C::STAGES; ++s) {
                ptx::mbar_init(BREADY0 + 8u * s, 4 * CG);   // converter warps of the group
                ptx::mbar_init(PFULL0 + 8u * s, 1);
            }
        }
        *abort_flag = 0;
        ptx::fence_mbar_init();
        ptx::fence_proxy_async_smem();
    }
    if (warp == 1) {
        if constexpr (CG == 2) {
            ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), C::TMEM_COLS);
            ptx::tmem_relinquish_pair();
        } else {
            ptx::tmem_alloc(ptx::smem_u32(tmem_slot), C::TMEM_COLS);
            ptx::tmem_relinquish();
        }
    }
    ptx::tc_fence_before();
    if constexpr (CG == 2) ptx::cluster_sync(); else __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // With TMEM allocated in every CTA of the grid, a dependent small kernel (a reduce,
    // AdamW) may launch and wait for this grid on the SMs it leaves free.  The wait is
    // a no-op here (the GEMMs are launched with full stream serialization); it stays so
    // that the kernel is correct under any launch.
    ptx::pdl_trigger();
    ptx::pdl_wait();
    if (threadIdx.x == 32) atomicAdd(&g_gemm_count[1], 1ull);

    uint32_t issued = 0, issued_parity = 0;   // producer: stages with a copy issued, and its phase
    if (warp == 0 && lane == 0) {
        // ------------------------------------------------------------ TMA producer
        for (int p = 0; p < grp.count; ++p) {
            ptx::tma_prefetch_desc(&grp.mA[p]);
            ptx::tma_prefetch_desc(&grp.mB0[p]);
            if (C::NB == 2 || C::F8) ptx::tma_prefetch_desc(&grp.mB1[p]);
            if constexpr (C::F8) ptx::tma_prefetch_desc(&grp.mA1[p]);
        }
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int ug = unit; ok && ug < total_units; ug += units) {
            const int p = group_find(grp, ug);
            const GemmArgs& a = grp.args[p];
            const int u = ug - grp.unit_begin[p];
            const CUtensorMap* tmA = &grp.mA[p];
            const CUtensorMap* tmB0 = &grp.mB0[p];
            const CUtensorMap* tmB1 = &grp.mB1[p];
            int mt, nt;
            tile_coords<C::RASTER>(a.tile_begin + u / a.split, a.tiles_m, a.tiles_n, mt, nt);
            const int arow = mt * C::TILE_M + static_cast<int>(rank) * kBM;
            const int brow = nt * C::BN + static_cast<int>(rank) * C::B_ROWS;
            const int kb0 = (u % a.split) * a.kb_per, kb1 = min(a.num_kb, kb0 + a.kb_per);
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!wait_bounded(EMPTY0 + 8u * stage, phase ^ 1u, abort_flag, true, SITE + 1)) {
                    ok = false;
                    break;
                }
                const uint32_t full = FULL0 + 8u * stage;
                // the pair's copies all count on the leader's barrier
                const uint32_t full_at = CG == 2 ? ptx::mapa_shared(full, 0) : full;
                const uint32_t sA = base + stage * C::STAGE_BYTES;
                const uint32_t sB0 = sA + C::A_BYTES;
                if (rank == 0) ptx::mbar_arrive_expect_tx(full, C::TX_BYTES);
                auto load = [&](uint32_t dst, const CUtensorMap* m, int x, int y) {
                    if constexpr (CG == 2) ptx::tma_load_2d_pair(dst, m, x, y, full_at);
                    else ptx::tma_load_2d(dst, m, x, y, full_at);
                };
                const int k0 = kb * C::BK;
                if constexpr (C::PK) {   // this CTA's B rows as 2-bit codes, for its converters
                    const uint32_t pfull = PFULL0 + 8u * stage;
                    ptx::mbar_arrive_expect_tx(pfull, C::P_BYTES);
                    if constexpr (C::EPI == EPI_DX)   // K-major: rows of W, 16 contraction codes per word
                        ptx::tma_load_2d(pring0 + stage * C::P_BYTES, tmB0, k0 / 16, brow, pfull);
                    else
                        ptx::tma_load_2d(pring0 + stage * C::P_BYTES, tmB0, brow / 16, k0, pfull);
                }
                if constexpr (C::A_MN) {
#pragma unroll
                    for (int j = 0; j < kBM / 64; ++j) load(sA + j * 64 * C::BK * 2, tmA, arow + j * 64, k0);
                } else {
                    load(sA, tmA, k0, arow);
                }
#pragma unroll
                for (int b = 0; b < (C::PK ? 0 : C::NB); ++b) {
                    const CUtensorMap* tmB = b == 0 ? tmB0 : tmB1;
                    const uint32_t sB = sB0 + b * C::B_BYTES;
                    if constexpr (C::B_MN) {
#pragma unroll
                        for (int j = 0; j < C::B_ROWS / 64; ++j) load(sB + j * 64 * C::BK * 2, tmB, brow + j * 64, k0);
                    } else {
                        load(sB, tmB, k0, brow);
                    }
                }
                if constexpr (C::F8) {   // the e4m3 halves: A8 rows of BK bytes, then B8
                    const uint32_t sA8 = sB0 + C::B_BYTES;
                    load(sA8, &grp.mA1[p], k0, arow);
                    load(sA8 + C::A8_BYTES, tmB1, k0, brow);
                }
                issued |= 1u << stage;
                issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        // Producer tail: wait until the MMA has released every stage filled above.  The
        // release is an asynchronous arrival (multicast to both CTAs of a pair) that may
        // otherwise land after this CTA has exited, in the barriers of the next CTA
        // placed on this SM.
        if (ok) {
            for (int s = 0; s < C::STAGES; ++s)
                if (issued & (1u << s))
                    wait_bounded(EMPTY0 + 8u * s, (issued_parity >> s) & 1u, abort_flag, true, SITE + 2);
        }
    } else if (warp == 1 && lane == 0 && rank == 0) {
        // ------------------------------------------------------------ MMA issuer (leader only)
        // bf16 operands, or binary16 (F8's first pass: kind::f16 with format code 0)
        constexpr uint32_t IDESC = make_idesc(C::TILE_M, C::BN, C::A_MN, C::B_MN, C::F8 ? 0u : 1u);
        constexpr uint32_t IDESC8 = make_idesc(C::TILE_M, C::BN, false, false, 0u);   // kind::f8f6f4, e4m3 x e4m3
        auto mma = [&](uint32_t d, uint64_t da, uint64_t db, uint32_t acc) {
            if constexpr (CG == 2) ptx::mma_bf16_pair(d, da, db, IDESC, acc);
            else ptx::mma_bf16(d, da, db, IDESC, acc);
        };
        auto mma8 = [&](uint32_t d, uint64_t da, uint64_t db) {
            if constexpr (CG == 2) ptx::mma_f8_pair(d, da, db, IDESC8, 1u);
            else ptx::mma_f8(d, da, db, IDESC8, 1u);
        };
        auto commit_all = [&](uint32_t bar) {   // arrive on `bar` in every CTA of the group
            if constexpr (CG == 2) ptx::mma_commit_pair_mc(bar, 0x3);
            else ptx::mma_commit(bar);
        };
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        int local = 0;
        for (int ug = unit; ok && ug < total_units; ug += units, ++local) {
            const int p = group_find(grp, ug);
            const GemmArgs& a = grp.args[p];
            const int u = ug - grp.unit_begin[p];
            const int acc = local & 1;
            const uint32_t acc_parity = (local >> 1) & 1;
            if (!wait_bounded(TEMPTY0 + 8u * acc, acc_parity ^ 1u, abort_flag, true, SITE + 3)) break;
            ptx::tc_fence_after();
            const uint32_t d_tmem = tmem_base + acc * C::BN;
            const int kb0 = (u % a.split) * a.kb_per, kb1 = min(a.num_kb, kb0 + a.kb_per);
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!wait_bounded(FULL0 + 8u * stage, phase, abort_flag, true, SITE + 4)) {
                    ok = false;
                    break;
                }
                if (C::PK && !wait_bounded(BREADY0 + 8u * stage, phase, abort_flag, true, SITE + 4)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t sA = base + stage * C::STAGE_BYTES;
                const uint32_t sB0 = sA + C::A_BYTES;
#pragma unroll
                for (int kk = 0; kk < C::BK / 16; ++kk) {
                    const uint64_t da = op_desc<C::A_MN, C::BK>(sA, kk);
                    mma(d_tmem, da, op_desc<C::B_MN, C::BK>(sB0, kk), (kb != kb0 || kk != 0) ? 1u : 0u);
                    if constexpr (C::NB == 2) mma(d_tmem, da, op_desc<C::B_MN, C::BK>(sB0 + C::B_BYTES, kk), 1u);
                }
                if constexpr (C::F8) {
                    // the e4m3 pass: rows of 64 bytes (SW64), 32-deep k-slices 32 bytes apart,
                    // into the same accumulator
                    const uint32_t sA8 = sB0 + C::B_BYTES, sB8 = sA8 + C::A8_BYTES;
#pragma unroll
                    for (int kk = 0; kk < C::BK / 32; ++kk)
                        mma8(d_tmem, make_sdesc(sA8 + kk * 32u, 16u, 512u, SW64), make_sdesc(sB8 + kk * 32u, 16u, 512u, SW64));
                }
                commit_all(EMPTY0 + 8u * stage);   // frees the stage once these MMAs are done
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            commit_all(TFULL0 + 8u * acc);          // accumulator ready for the epilogue
        }
        // every MMA this thread issued completes before TMEM and shared memory go away
        if constexpr (CG == 2) ptx::mma_commit_pair(DRAIN); else ptx::mma_commit(DRAIN);
        wait_bounded(DRAIN, 0, abort_flag, false, SITE + 5);
        // Accumulator tail: wait for the epilogues' release of the last use of each
        // accumulator, so that the peer CTA's remote arrivals have landed before exit.
        if (ok && !*abort_flag) {
            for (int acc = 0; acc < 2; ++acc) {
                if (local <= acc) continue;
                const int last = (local - 1) - (((local - 1) - acc) & 1);   // last unit that used acc
                wait_bounded(TEMPTY0 + 8u * acc, static_cast<uint32_t>(last >> 1) & 1u, abort_flag, true, SITE + 6);
            }
        }
    } else if (C::PK && warp >= 2 + C::EPI_WARPS) {
        // ------------------------------------------------------------ operand converters
        // The producer copies each stage's B rows as 2-bit codes (TMA, P_BYTES) into this
        // CTA's ring; thread ct takes k-row ct/2 and half ct&1 of those rows (WPT words of 16
        // columns), expands them into the swizzled MN-major bf16 layout a TMA copy of T
        // would have written (64-column chunks of 64 k-rows x 128 B), and the warps signal
        // the MMA issuer.  The stage is free when its codes land: the producer copies them
        // only after the stage's release.
        constexpr int WPT = C::B_ROWS / 32;
        const int team = (warp - 2 - C::EPI_WARPS) >> 2;   // team t takes the k-blocks of running index t mod 2
        const int ct = static_cast<int>(threadIdx.x) - 32 * (2 + C::EPI_WARPS) - 128 * team;
        const int kr = ct >> 1, half = ct & 1;
        const uint32_t bready_peer = CG == 2 ? ptx::mapa_shared(BREADY0, 0) : BREADY0;
        int stage = 0;
        uint32_t phase = 0;
        int seq = 0;   // running k-block index over this CTA's units
        for (int ug = unit; ug < total_units; ug += units) {
            const int p = group_find(grp, ug);
            const GemmArgs& a = grp.args[p];
            const int u = ug - grp.unit_begin[p];
            const int kb0 = (u % a.split) * a.kb_per, kb1 = min(a.num_kb, kb0 + a.kb_per);
            bool ok = true;
            for (int kb = kb0; kb < kb1; ++kb, ++seq) {
                if ((seq & 1) != team) {   // the other team's k-block: only follow the stage ring
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    continue;
                }
                const bool landed = wait_bounded(PFULL0 + 8u * stage, phase, abort_flag, true, SITE + 9);
                if (!__all_sync(0xffffffffu, landed)) {
                    ok = false;
                    break;
                }
                if constexpr (C::EPI == EPI_DX) {
                    // K-major W_hi / W_lo: this thread's rows of W (ct, ct + 128, ...), each 64
                    // contraction indices as four words of 16 codes; a 16-byte unit holds eight
                    // consecutive indices c as bf16 pairs t*s_hi[c], t*s_lo[c] (the sign bit flipped
                    // for t = -1, +0 for t = 0: the bits tern_materialize writes)
                    const uint16_t* shi = reinterpret_cast<const uint16_t*>(a.packed);   // s_hi [Kg], s_lo after
                    const uint16_t* slo = shi + a.Kg;
                    const int c0 = kb * C::BK;
                    const uint32_t sB = base + stage * C::STAGE_BYTES + C::A_BYTES;
#pragma unroll
                    for (int rr = 0; rr < C::B_ROWS / 128; ++rr) {
                        const int r = ct + 128 * rr;
                        uint32_t w[4];
                        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                     : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                                     : "r"(pring0 + stage * C::P_BYTES + static_cast<uint32_t>(r) * 16u)
                                     : "memory");
                        const uint32_t rowoff = static_cast<uint32_t>(r >> 3) * 1024u + static_cast<uint32_t>(r & 7) * 128u;
#pragma unroll
                        for (int un = 0; un < 8; ++un) {
                            uint4 h4 = make_uint4(0u, 0u, 0u, 0u), l4 = h4;
                            if (c0 + 8 * un < a.Kg) {   // Kg % 16 == 0: the unit is wholly inside or outside
                                h4 = __ldg(reinterpret_cast<const uint4*>(shi + c0 + 8 * un));
                                l4 = __ldg(reinterpret_cast<const uint4*>(slo + c0 + 8 * un));
                            }
                            const uint32_t hp[4] = {h4.x, h4.y, h4.z, h4.w}, lp[4] = {l4.x, l4.y, l4.z, l4.w};
                            const uint32_t w16 = w[un >> 1] >> (16 * (un & 1));
                            uint32_t qh[4], ql[4];
#pragma unroll
                            for (int pr = 0; pr < 4; ++pr) {
                                const uint32_t x = (w16 >> (4 * pr)) & 0xFu;   // codes of c and c + 1
                                const uint32_t nz = ((x & 1u) | ((x & 4u) << 14)) * 0xFFFFu;
                                const uint32_t ng = ((x & 2u) << 14) | ((x & 8u) << 28);
                                qh[pr] = (hp[pr] & nz) ^ ng;
                                ql[pr] = (lp[pr] & nz) ^ ng;
                            }
                            const uint32_t at = rowoff + (static_cast<uint32_t>(un ^ (r & 7)) << 4);
                            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sB + at), "r"(qh[0]),
                                         "r"(qh[1]), "r"(qh[2]), "r"(qh[3])
                                         : "memory");
                            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sB + C::B_BYTES + at),
                                         "r"(ql[0]), "r"(ql[1]), "r"(ql[2]), "r"(ql[3])
                                         : "memory");
                        }
                    }
                } else {
                const uint32_t src = pring0 + stage * C::P_BYTES + static_cast<uint32_t>(kr) * (C::B_ROWS / 16) * 4u +
                                     static_cast<uint32_t>(half) * WPT * 4u;
                const uint32_t sB = base + stage * C::STAGE_BYTES + C::A_BYTES;
#pragma unroll
                for (int h = 0; h < WPT / 4; ++h) {
                    uint32_t w[4];
                    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                                 : "r"(src + h * 16u)
                                 : "memory");
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int col = (half * WPT + 4 * h + j) * 16;   // first column of the word in the CTA's rows
                        const uint32_t row = sB + (col >> 6) * (64u * C::BK * 2u) + static_cast<uint32_t>(kr) * 128u;
                        const int u0 = (col & 63) >> 3;                 // its first 16-byte unit in the row
                        uint32_t q[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) q[i] = tern_pair_bf16(w[j] >> (2 * i));
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                                         row + (static_cast<uint32_t>(u0 ^ (kr & 7)) << 4)),
                                     "r"(q[0]), "r"(q[1]), "r"(q[2]), "r"(q[3])
                                     : "memory");
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                                         row + (static_cast<uint32_t>((u0 + 1) ^ (kr & 7)) << 4)),
                                     "r"(q[4]), "r"(q[5]), "r"(q[6]), "r"(q[7])
                                     : "memory");
                    }
                }
                }
                ptx::fence_proxy_async_smem();   // generic-proxy writes, read next by the tensor core
                __syncwarp();
                if (lane == 0) {
                    if (CG == 2 && rank != 0) ptx::mbar_arrive_cluster(bready_peer + 8u * stage);
                    else ptx::mbar_arrive(BREADY0 + 8u * stage);
                }
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
        }
    } else if (warp >= 2 && warp < 2 + C::EPI_WARPS) {
        // ------------------------------------------------------------ epilogue
        const int quad = warp & 3;   // a warp may touch TMEM lanes 32*(warp%4) .. +31
        const uint32_t tempty_leader = CG == 2 ? ptx::mapa_shared(TEMPTY0, 0) : TEMPTY0;
        // with eight epilogue warps, warps 2-5 take the tile's first BN/2 columns and 6-9 the rest
        constexpr int JPW = C::BN / 32 / (C::EPI_WARPS / 4);   // 32-column chunks per warp and tile
        const int j0 = ((warp - 2) / 4) * JPW;
        int local = 0;
        // the column scales of a unit's tile (none for dX and for split units' raw tiles)
        auto unit_scales = [&](int ugn, float (&sc)[8]) {
            const float* sp = nullptr;
            int col0 = 0, ng = 0;
            if (C::EPI != EPI_DX && ugn < total_units) {
                const int pn = group_find(grp, ugn);
                const GemmArgs& an = grp.args[pn];
                if (an.partial_g == nullptr && (C::EPI == EPI_FWD || an.out != nullptr)) {
                    int mtn, ntn;
                    tile_coords<C::RASTER>(an.tile_begin + (ugn - grp.unit_begin[pn]) / an.split, an.tiles_m,
                                         an.tiles_n, mtn, ntn);
                    sp = an.scale;
                    col0 = ntn * C::BN;
                    ng = an.Ng;
                }
            }
            load_tile_scales(sp, col0, ng, lane, sc);
        };
        float sc_cur[8], sc_next[8];
        unit_scales(unit, sc_cur);
        for (int ug = unit; ug < total_units; ug += units, ++local) {
            const int p = group_find(grp, ug);
            const GemmArgs& a = grp.args[p];
            const int u = ug - grp.unit_begin[p];
            const int acc = local & 1;
            const uint32_t acc_parity = (local >> 1) & 1;
            // one decision per warp: the loads below are warp-collective
            const bool full = wait_bounded(TFULL0 + 8u * acc, acc_parity, abort_flag, true, SITE + 7);
            if (!__all_sync(0xffffffffu, full)) break;
            ptx::tc_fence_after();
            unit_scales(ug + units, sc_next);   // in flight while this tile drains
            int mt, nt;
            tile_coords<C::RASTER>(a.tile_begin + u / a.split, a.tiles_m, a.tiles_n, mt, nt);
            const int row0 = mt * C::TILE_M + static_cast<int>(rank) * kBM;
            const uint32_t trow = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * C::BN;
            if (C::EPI == EPI_DW && a.partial_g != nullptr) {
                // split unit: the raw partial tile (row-major TILE_M x BN, unit after unit in
                // partial_g) for the reduce kernel
                float* pg = a.partial_g + (static_cast<int64_t>(u) * C::TILE_M + static_cast<int>(rank) * kBM + quad * 32) *
                                              C::BN;
#pragma unroll 1
                for (int j = j0; j < j0 + JPW; ++j) {
                    uint32_t r[32];
                    ptx::tmem_ld_32x32b_x32(trow + j * 32, r);
                    ptx::tmem_wait_ld();
                    float v[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
                    store_chunk(pg + j * 32, C::BN, 32, 32, v, false, lane);
                }
            } else if (row0 < a.Mg) {   // a pair's second half may lie wholly past the last row
                const int tile128 = mt * CG + static_cast<int>(rank);
                const int wrow = row0 + quad * 32;
                const int rexp = C::F8 && wrow + lane < a.Mg ? __ldg(a.row_exp + wrow + lane) : 0;
#pragma unroll 1
                for (int j = j0; j < j0 + JPW; ++j) {
                    const int c0 = nt * C::BN + j * 32;
                    if (c0 >= a.Ng) break;
                    uint32_t r[32];
                    ptx::tmem_ld_32x32b_x32(trow + j * 32, r);
                    ptx::tmem_wait_ld();
                    epilogue_chunk<C>(a, r, sc_cur, j, wrow + lane, wrow, c0, tile128, quad, lane, rexp);
                }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) sc_cur[i] = sc_next[i];
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if constexpr (CG == 2) ptx::mbar_arrive_cluster(tempty_leader + 8u * acc);
                else ptx::mbar_arrive(TEMPTY0 + 8u * acc);
            }
        }
    }

    ptx::tc_fence_before();
    if constexpr (CG == 2) ptx::cluster_sync(); else __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        if constexpr (CG == 2) ptx::tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
        else ptx::tmem_dealloc(tmem_base, C::TMEM_COLS);
        if (lane == 0) atomicAdd(&g_gemm_count[2], 1ull);
    }
    if (warp == 0 && lane == 0 && *abort_flag) {
        // after an abort, copies still in flight must land before the CTA's shared memory is released
        if constexpr (CG == 1) {
            for (int s = 0; s < C::STAGES; ++s)
                if (issued & (1u << s)) {
                    wait_bounded(FULL0 + 8u * s, (issued_parity >> s) & 1u, abort_flag, false, SITE + 8);
                    if constexpr (C::PK)
                        wait_bounded(PFULL0 + 8u * s, (issued_parity >> s) & 1u, abort_flag, false, SITE + 8);
                }
        } else {
            // a pair's copies complete on the leader's barriers; give them time to land
            const uint64_t t0 = ptx::globaltimer();
            while (ptx::globaltimer() - t0 < 100000ull) {
            }
        }
    }
}

}  // namespace

// One launch runs the work units of a group of G problems (G = 1: a single
// layer); the tensor maps live in the kernel's parameter space.
template <int CG, int G>
__global__ void __launch_bounds__(320, 1) tern_fwd_gemm(const __grid_constant__ GemmGroup<G> grp) {
    gemm_body<std::conditional_t<CG == 2, Fwd2, Fwd1>>(grp);
}

// The forward with T read as 2-bit codes (expanded in shared memory by converter warps).
template <int CG, int G>
__global__ void __launch_bounds__(448, 1) tern_fwdp_gemm(const __grid_constant__ GemmGroup<G> grp) {
    gemm_body<std::conditional_t<CG == 2, FwdP2, FwdP1>>(grp);
}

template <int CG, int G>
__global__ void __launch_bounds__(320, 1) tern_dx_gemm(const __grid_constant__ GemmGroup<G> grp) {
    gemm_body<std::conditional_t<CG == 2, Dx2, Dx1>>(grp);
}

template <int CG, int G>
__global__ void __launch_bounds__(320, 1) tern_dw_gemm(const __grid_constant__ GemmGroup<G> grp) {
    gemm_body<std::conditional_t<CG == 2, Dw2, Dw1>>(grp);
}

// dX with W_hi / W_lo expanded from the 2-bit codes inside the GEMM (converter warps, as
// the forward's tern_fwdp_gemm) and a per-column s_hi / s_lo table.
template <int CG, int G>
__global__ void __launch_bounds__(448, 1) tern_dxp_gemm(const __grid_constant__ GemmGroup<G> grp) {
    gemm_body<std::conditional_t<CG == 2, DxP2, DxP1>>(grp);
}

// dX from the fp16 + e4m3 split (split8.cu): a binary16 pass and an e4m3 pass into one
// accumulator, the dY row exponent applied in the epilogue.
template <int CG, int G>
__global__ void __launch_bounds__(320, 1) tern_dx8_gemm(const __grid_constant__ GemmGroup4<G> grp) {
    gemm_body<std::conditional_t<CG == 2, Dx8_2, Dx8_1>>(grp);
}

// Self-test of the bounded wait: one warp waits on an mbarrier that nothing
// arrives on, with the GEMMs' wait routine and a short limit; it must give up,
// record TERN_ERR_TIMEOUT and return.
__global__ void tern_wait_selftest(uint64_t limit_ns) {
    ptx::pdl_trigger();
    ptx::pdl_wait();
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        ptx::mbar_init(ptx::smem_u32(&bar), 1);
        abort_flag = 0;
        ptx::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) wait_bounded(ptx::smem_u32(&bar), 0, &abort_flag, false, 999, limit_ns);
}

// sum_i partial[i][c] in ascending i; eight loads go out before their (ordered) adds.
__device__ __forceinline__ float ordered_column_sum(const float* __restrict__ partial, int nparts, int N, int c) {
    float s = 0.0f;
    int i = 0;
    for (; i + 8 <= nparts; i += 8) {
        float x[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) x[k] = partial[static_cast<int64_t>(i + k) * N + c];
#pragma unroll
        for (int k = 0; k < 8; ++k) s += x[k];
    }
    for (; i < nparts; ++i) s += partial[static_cast<int64_t>(i) * N + c];
    return s;
}

// sgrad[c] = sum over the partial rows in ascending order (deterministic); with
// accumulate, that sum is added to the stored sgrad[c].
__global__ void tern_sgrad_reduce(const float* __restrict__ partial, int nparts, int N, float* __restrict__ sgrad,
                                  int accumulate) {
    ptx::pdl_trigger();
    ptx::pdl_wait();
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= N) return;
    sgrad[c] = accumulate ? sgrad[c] + ordered_column_sum(partial, nparts, N, c) : ordered_column_sum(partial, nparts, N, c);
}

// The split tiles of up to G problems: problem p owns blocks [block_begin[p], block_begin[p+1]).
template <int G>
struct ReduceGroup {
    GemmArgs args[G];
    int block_begin[G + 1];
    int count;
    int tile_m, tile_n;
};

// Finish the split G tiles: G = sum over the tile's slices in slice order, then the
// same epilogue as the G kernel (gq = G*scale[c], or += with accumulate, and the sgrad
// partial of each 32-row group).  One CTA per 32-row group and 128-column half of a
// tile: warp w takes rows 4w..4w+3 of the group, lane l columns 4l..4l+3 of the half
// (16-byte loads: a warp reads 512 contiguous bytes of a row; two slices' loads go out
// before their adds); the eight warps' column sums are added in warp order through
// shared memory.
template <int G>
__global__ void __launch_bounds__(256) tern_dw_split_reduce(const __grid_constant__ ReduceGroup<G> grp) {
    ptx::pdl_trigger();
    ptx::pdl_wait();
    int p = 0;
    while (p + 1 < grp.count && static_cast<int>(blockIdx.x) >= grp.block_begin[p + 1]) ++p;
    const GemmArgs& a = grp.args[p];
    const int block = static_cast<int>(blockIdx.x) - grp.block_begin[p];
    const int tile_m = grp.tile_m, tile_n = grp.tile_n;
    const int halves = tile_n / 128;
    const int per_tile = (tile_m / 32) * halves;
    const int j = block / per_tile;                        // split tile
    const int rg = (block % per_tile) / halves;            // 32-row group within the tile
    const int hf = block % halves;                         // 128-column half within the tile
    int tm, tn;
    if (tile_m == 2 * kBM) tile_coords<8>(a.tile_begin + j, a.tiles_m, a.tiles_n, tm, tn);
    else tile_coords<16>(a.tile_begin + j, a.tiles_m, a.tiles_n, tm, tn);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c_in = hf * 128 + lane * 4;                  // first of this thread's columns in the tile
    const int col = tn * tile_n + c_in;
    const int r_base = tm * tile_m + rg * 32;
    // partial rows exist for every 32-row group of the 128-row blocks that hold rows;
    // a group wholly past the last row still writes its (zero) partial
    if (r_base >= ((a.Mg + kBM - 1) / kBM) * kBM) return;
    const bool col_ok = col < a.Ng;                        // N % 16 == 0: all four columns or none
    const int64_t tile_elems = static_cast<int64_t>(tile_m) * tile_n;
    const float* base = a.partial_g + static_cast<int64_t>(j) * a.split * tile_elems +
                        static_cast<int64_t>(rg * 32 + warp * 4) * tile_n + c_in;
    float4 g[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) g[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    auto add = [](float4& s, const float4& x) {
        s.x += x.x;
        s.y += x.y;
        s.z += x.z;
        s.w += x.w;
    };
    int sl = 0;
    for (; sl + 2 <= a.split; sl += 2) {
        float4 x0[4], x1[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x0[i] = __ldcs(reinterpret_cast<const float4*>(base + sl * tile_elems + i * tile_n));
            x1[i] = __ldcs(reinterpret_cast<const float4*>(base + (sl + 1) * tile_elems + i * tile_n));
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            add(g[i], x0[i]);
            add(g[i], x1[i]);
        }
    }
    if (sl < a.split) {
#pragma unroll
        for (int i = 0; i < 4; ++i) add(g[i], __ldcs(reinterpret_cast<const float4*>(base + sl * tile_elems + i * tile_n)));
    }
    float cs[4] = {0.f, 0.f, 0.f, 0.f};
    if (col_ok) {
        const float4 sc = a.out ? *reinterpret_cast<const float4*>(a.scale + col) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int row = r_base + warp * 4 + i;
            if (row >= a.Mg) break;
            if (a.out) {
                float4 v = make_float4(g[i].x * sc.x, g[i].y * sc.y, g[i].z * sc.z, g[i].w * sc.w);
                float4* o = reinterpret_cast<float4*>(a.out + static_cast<int64_t>(row) * a.Ng + col);
                if (a.accumulate) {
                    const float4 old = *o;
                    v = make_float4(old.x + v.x, old.y + v.y, old.z + v.z, old.w + v.w);
                }
                *o = v;
            }
            if (a.partial) {
                const uint32_t w = a.packed[static_cast<int64_t>(row) * (a.Ng / 16) + col / 16] >> (2 * (col % 16));
                const float gv[4] = {g[i].x, g[i].y, g[i].z, g[i].w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t code = (w >> (2 * k)) & 3u;
                    cs[k] += (code & 1u) ? ((code & 2u) ? -gv[k] : gv[k]) : 0.0f;
                }
            }
        }
    }
    if (a.partial == nullptr) return;
    __shared__ float red[8][128];
#pragma unroll
    for (int k = 0; k < 4; ++k) red[warp][lane * 4 + k] = cs[k];
    __syncthreads();
    if (threadIdx.x < 128) {
        const int cc = tn * tile_n + hf * 128 + static_cast<int>(threadIdx.x);
        if (cc < a.Ng) {
            float s = 0.0f;
#pragma unroll
            for (int w = 0; w < 8; ++w) s += red[w][threadIdx.x];
            a.partial[static_cast<int64_t>(r_base / 32) * a.Ng + cc] = s;
        }
    }
}

// ===================================================================== host side

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Encoded tensor maps, cached per process: a map depends only on the address, the
// element type, the extents, the box and the swizzle (not on the device or stream),
// so a call that repeats a layer's buffers (every training step) reuses its maps
// instead of encoding them again on the host.  Direct-mapped, 1024 entries.
struct MapKey {
    const void* ptr;
    int64_t inner, outer;
    int box_inner, box_outer, sw, dtype;
    bool operator==(const MapKey& o) const {
        return ptr == o.ptr && inner == o.inner && outer == o.outer && box_inner == o.box_inner &&
               box_outer == o.box_outer && sw == o.sw && dtype == o.dtype;
    }
};
struct MapSlot {
    MapKey key;
    CUtensorMap map;
    bool valid;
};
constexpr int kMapCache = 1024;
MapSlot g_map_cache[kMapCache];
std::mutex g_map_mu;

int encode_2d(CUtensorMap* m, const MapKey& k) {
    size_t h = reinterpret_cast<uintptr_t>(k.ptr) >> 4;
    h ^= static_cast<size_t>(k.inner) * 0x9E3779B97F4A7C15ull ^ static_cast<size_t>(k.outer) * 0xC2B2AE3D27D4EB4Full;
    h ^= static_cast<size_t>(k.box_inner * 131 + k.box_outer * 7 + k.sw * 3 + k.dtype) * 0x165667B19E3779F9ull;
    MapSlot& slot = g_map_cache[(h ^ (h >> 29)) % kMapCache];
    {
        std::lock_guard<std::mutex> lock(g_map_mu);
        if (slot.valid && slot.key == k) {
            *m = slot.map;
            return TERN_OK;
        }
    }
    EncodeTiledFn enc = encode_fn();
    if (!enc) return TERN_ERR_CUDA;
    const int esize = (k.dtype == CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 || k.dtype == CU_TENSOR_MAP_DATA_TYPE_FLOAT16) ? 2
                      : k.dtype == CU_TENSOR_MAP_DATA_TYPE_UINT8                                              ? 1
                                                                                                              : 4;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(k.inner), static_cast<cuuint64_t>(k.outer)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(k.inner) * esize};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(k.box_inner), static_cast<cuuint32_t>(k.box_outer)};
    cuuint32_t estr[2] = {1, 1};
    // operands are read with 256-byte L2 promotion; outputs are only written
    const CUtensorMapL2promotion l2 =
        k.dtype == CU_TENSOR_MAP_DATA_TYPE_FLOAT32 ? CU_TENSOR_MAP_L2_PROMOTION_NONE : CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
    CUresult r = enc(m, static_cast<CUtensorMapDataType>(k.dtype), 2, const_cast<void*>(k.ptr), dims, strides, box,
                     estr, CU_TENSOR_MAP_INTERLEAVE_NONE, static_cast<CUtensorMapSwizzle>(k.sw), l2,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return TERN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_map_mu);
    slot.key = k;
    slot.map = *m;
    slot.valid = true;
    return TERN_OK;
}

// Tensor map of a row-major bf16 matrix [outer][inner] read in boxes of box_outer x box_inner.
int map_bf16(CUtensorMap* m, const void* ptr, int64_t inner, int64_t outer, int box_inner, int box_outer,
             CUtensorMapSwizzle sw) {
    return encode_2d(m, MapKey{ptr, inner, outer, box_inner, box_outer, static_cast<int>(sw),
                               static_cast<int>(CU_TENSOR_MAP_DATA_TYPE_BFLOAT16)});
}

// Boxes of one operand: K-major tiles are read as one box of BK x rows; MN-major
// tiles as 64-wide boxes of BK k-rows.
template <class C>
int map_operand(CUtensorMap* m, const void* ptr, int64_t inner, int64_t outer, bool mn, int rows) {
    const CUtensorMapSwizzle sw = C::BK == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    return mn ? map_bf16(m, ptr, inner, outer, 64, C::BK, sw) : map_bf16(m, ptr, inner, outer, C::BK, rows, sw);
}

template <class C>
GemmArgs make_args(int64_t Mg, int64_t Ng, int64_t Kg) {
    GemmArgs a{};
    a.Mg = static_cast<int>(Mg);
    a.Ng = static_cast<int>(Ng);
    a.Kg = static_cast<int>(Kg);
    a.tiles_m = static_cast<int>((Mg + C::TILE_M - 1) / C::TILE_M);
    a.tiles_n = static_cast<int>((Ng + C::BN - 1) / C::BN);
    a.num_tiles = a.tiles_m * a.tiles_n;
    a.num_kb = static_cast<int>((Kg + C::BK - 1) / C::BK);
    a.tile_begin = 0;
    a.num_units = a.num_tiles;
    a.split = 1;
    a.kb_per = a.num_kb;
    a.partial_g = nullptr;
    return a;
}

// Co-resident CTA pairs (or CTAs) of a GEMM kernel: the persistent grid.  Sets
// the kernel's shared-memory attribute once per device, so later calls (e.g.
// under stream capture) only enqueue launches.
template <class C, class K>
int persistent_units(K kernel, int num_sms, int* units) {
    static std::once_flag once[64];
    static cudaError_t attr_status[64];
    static int max_clusters[64];
    int dev = 0;
    TERN_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return TERN_ERR_DEVICE;
    std::call_once(once[dev], [&] {
        attr_status[dev] = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (attr_status[dev] != cudaSuccess || C::CG == 1) return;
        cudaLaunchConfig_t cfg{};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(2 * (num_sms / 2));
        cfg.blockDim = dim3(C::THREADS);
        cfg.dynamicSmemBytes = C::SMEM_BYTES;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        attr_status[dev] = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg);
        max_clusters[dev] = n > 0 ? n : 1;
    });
    TERN_CUDA_TRY(attr_status[dev]);
    *units = C::CG == 2 ? max_clusters[dev] : num_sms;
    return TERN_OK;
}

// Persistent launch of a problem group: one CTA (or CTA pair) per SM (pair of
// SMs), at most one per work unit.  No programmatic stream serialization: the grid
// starts once every earlier kernel on the stream has completed, so its TMEM
// allocation and cluster barrier (waits without a bound) never wait on another grid.
template <class C, class K, class GRP>
int launch(K kernel, const GRP& grp, int num_sms, cudaStream_t s) {
    int units = 0;
    if (int st = persistent_units<C>(kernel, num_sms, &units)) return st;
    const int total = grp.unit_begin[grp.count];
    if (total <= 0) return TERN_OK;
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = C::CG == 2 ? 1 : 0;
    cfg.gridDim = dim3(C::CG * std::min(total, units));
    TERN_CUDA_TRY(cudaLaunchKernelEx(&cfg, kernel, grp));
    return TERN_OK;
}

bool dims_ok(int64_t M, int64_t K, int64_t N) {
    return M >= 1 && K >= 16 && N >= 16 && M < (1ll << 31) && K < (1ll << 31) && N < (1ll << 31) &&
           M * K < (1ll << 40) && K * N < (1ll << 40) && M * N < (1ll << 40);
}

// A CTA pair per tile once the output has at least two 128-row blocks.
bool use_pair(int64_t Mg) { return Mg > kBM; }

// Fill problem p of a group with its maps and arguments.
template <class C, int G>
int group_set(GemmGroup<G>& g, int p, const void* A, int64_t a_inner, int64_t a_outer, const void* B0,
              const void* B1, int64_t b_inner, int64_t b_outer, const GemmArgs& a) {
    if (int st = map_operand<C>(&g.mA[p], A, a_inner, a_outer, C::A_MN, kBM)) return st;
    if constexpr (C::PK && C::EPI == EPI_DX) {   // W as 2-bit codes [Ng][Kg/16] words (K-major rows)
        if (int st = encode_2d(&g.mB0[p], MapKey{a.bpacked, a.Kg / 16, a.Ng, C::BK / 16, C::B_ROWS,
                                                 static_cast<int>(CU_TENSOR_MAP_SWIZZLE_NONE),
                                                 static_cast<int>(CU_TENSOR_MAP_DATA_TYPE_UINT32)}))
            return st;
    } else if constexpr (C::PK) {   // B as 2-bit codes [Kg][Ng/16] words, copied per stage for the converters
        if (int st = encode_2d(&g.mB0[p], MapKey{a.bpacked, a.Ng / 16, a.Kg, C::B_ROWS / 16, C::BK,
                                                 static_cast<int>(CU_TENSOR_MAP_SWIZZLE_NONE),
                                                 static_cast<int>(CU_TENSOR_MAP_DATA_TYPE_UINT32)}))
            return st;
    } else {
        if (int st = map_operand<C>(&g.mB0[p], B0, b_inner, b_outer, C::B_MN, C::B_ROWS)) return st;
    }
    if (B1) {
        if (int st = map_operand<C>(&g.mB1[p], B1, b_inner, b_outer, C::B_MN, C::B_ROWS)) return st;
    } else {
        g.mB1[p] = g.mB0[p];
    }
    g.args[p] = a;
    return TERN_OK;
}

// Unit ranges of the first `count` problems, from their num_units.
template <class GRP>
void group_close(GRP& g, int count) {
    g.count = count;
    g.unit_begin[0] = 0;
    for (int p = 0; p < count; ++p) g.unit_begin[p + 1] = g.unit_begin[p] + g.args[p].num_units;
}

template <class C, class K>
int run_fwd(K kernel, const uint16_t* X, const uint16_t* T, const uint32_t* packed, const float* scale, float* Y,
            int64_t M, int64_t K_, int64_t N, int num_sms, cudaStream_t s) {
    GemmGroup<1> g;
    GemmArgs a = make_args<C>(M, N, K_);
    a.out = Y;
    a.scale = scale;
    a.bpacked = C::PK ? packed : nullptr;
    if (int st = group_set<C>(g, 0, X, K_, M, C::PK ? nullptr : T, nullptr, N, K_, a)) return st;
    group_close(g, 1);
    return launch<C>(kernel, g, num_sms, s);
}

template <class C, class K>
int run_dx(K kernel, const uint16_t* dY, const uint16_t* whi, const uint16_t* wlo, float* dX, int64_t M,
           int64_t K_, int64_t N, int num_sms, cudaStream_t s) {
    GemmGroup<1> g;
    GemmArgs a = make_args<C>(M, K_, N);
    a.out = dX;
    if (int st = group_set<C>(g, 0, dY, N, M, whi, wlo, N, K_, a)) return st;
    group_close(g, 1);
    return launch<C>(kernel, g, num_sms, s);
}

// dX from the 2-bit codes [K][N/16] and the s_hi / s_lo table (hilo: N bf16 s_hi, then N s_lo).
template <class C, class K>
int run_dxp(K kernel, const uint16_t* dY, const uint32_t* codes, const uint16_t* hilo, float* dX, int64_t M,
            int64_t K_, int64_t N, int num_sms, cudaStream_t s) {
    GemmGroup<1> g;
    GemmArgs a = make_args<C>(M, K_, N);
    a.out = dX;
    a.bpacked = codes;
    a.packed = reinterpret_cast<const uint32_t*>(hilo);
    if (int st = group_set<C>(g, 0, dY, N, M, nullptr, nullptr, N, K_, a)) return st;
    group_close(g, 1);
    return launch<C>(kernel, g, num_sms, s);
}

// dX from the fp16 + e4m3 split: dY16 / dY8 [M][N] and the weight planes h*T / l*T [K][N].
template <class C, class K>
int run_dx8(K kernel, const uint16_t* dy16, const uint8_t* dy8, const int* row_exp, const uint16_t* wh16,
            const uint8_t* wl8, float* dX, int64_t M, int64_t K_, int64_t N, int num_sms, cudaStream_t s) {
    GemmGroup4<1> g;
    GemmArgs a = make_args<C>(M, K_, N);
    a.out = dX;
    a.row_exp = row_exp;
    auto map = [&](CUtensorMap* m, const void* ptr, int64_t outer, int rows, bool f16) {
        return encode_2d(m, MapKey{ptr, N, outer, 64, rows,
                                   static_cast<int>(f16 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B),
                                   static_cast<int>(f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8)});
    };
    if (int st = map(&g.mA[0], dy16, M, kBM, true)) return st;
    if (int st = map(&g.mB0[0], wh16, K_, C::B_ROWS, true)) return st;
    if (int st = map(&g.mA1[0], dy8, M, kBM, false)) return st;
    if (int st = map(&g.mB1[0], wl8, K_, C::B_ROWS, false)) return st;
    g.args[0] = a;
    group_close(g, 1);
    return launch<C>(kernel, g, num_sms, s);
}

// Largest number of split units the tail of a G launch may use (bounds the workspace).
constexpr int kMaxTailUnits = 128;
// ... and of a grouped G launch, whose split covers every tile of the group (at M = 8192
// the six RWKV-style projections have 48 G tiles of 128 k-blocks: split three ways they
// fill two waves of 76 pairs)
constexpr int kMaxGroupTailUnits = 256;

template <class C>
int64_t dw_tail_bytes(int64_t M, int64_t K_, int64_t N) {
    const GemmArgs a = make_args<C>(K_, N, M);
    const int64_t units = std::min<int64_t>(kMaxTailUnits, static_cast<int64_t>(a.num_tiles) * a.num_kb);
    return units * C::TILE_M * C::BN * static_cast<int64_t>(sizeof(float));
}

// G = X^T dY with the fused gq / sgrad epilogue.  Whole waves of tiles run as
// they are; when the last wave would leave units idle and `tail` has room, the
// remaining tiles are split along the token axis over the idle units and
// finished by tern_dw_split_reduce.
template <class C, int G>
int launch_split_reduce(const ReduceGroup<G>& r, cudaStream_t s) {
    return launch_pdl(tern_dw_split_reduce<G>, dim3(static_cast<unsigned>(r.block_begin[r.count])), dim3(256), 0, s,
                      r);
}

// G = X^T dY with the fused gq / sgrad epilogue.  Whole waves of tiles run as
// they are; when the last wave would leave units idle and `tail` has room, the
// remaining tiles are split along the token axis over the idle units and
// finished by tern_dw_split_reduce.
// The split factor of the tail of a G launch: the R tiles left after whole waves of
// `units` are split along the token axis into s slices of ceil(kb/s) k-blocks when that
// shortens the last rounds.  Minimises, in times of one 64-deep k-block of a 256 x 256
// tile, rounds(R*s) * ceil(kb/s) + 0.32 * R*s + 20: the reduce pass costs about 0.32 per
// partial tile and the extra launches about 20 (measured at the wide chain's G: 200
// partial tiles reduced in 17 us).
int tail_split(int R, int kb, int units, int max_units) {
    if (R <= 0) return 1;
    int best = 1;
    double best_cost = kb;   // one round of whole tiles
    for (int sp = 2; sp <= kb && R * sp <= max_units; ++sp) {
        const int per = (kb + sp - 1) / sp;
        const double cost = std::ceil(static_cast<double>(R) * sp / units) * per + 0.32 * R * sp + 20.0;
        if (cost < best_cost - 1e-9) {
            best = sp;
            best_cost = cost;
        }
    }
    return best;
}

// The G launch of one problem (index 0 of g): whole waves of tiles as they are; when the
// last wave would leave units idle and `tail` has room, its tiles are split along the
// token axis (tail_split) and finished by tern_dw_split_reduce.
template <class C, class K, class GRP>
int dw_waves_and_tail(K kernel, GRP& g, float* tail, int64_t tail_bytes, int max_units, int num_sms, cudaStream_t s) {
    if (tail) {
        int units = 0;
        if (int st = persistent_units<C>(kernel, num_sms, &units)) return st;
        const GemmArgs a = g.args[0];
        const int T = a.num_tiles, T0 = (T / units) * units, R = T - T0;
        int split = tail_split(R, a.num_kb, units, max_units);
        if (split >= 2) {
            const int kb_per = (a.num_kb + split - 1) / split;
            split = (a.num_kb + kb_per - 1) / kb_per;   // every slice non-empty
            const int64_t need = static_cast<int64_t>(R) * split * C::TILE_M * C::BN * sizeof(float);
            if (need <= tail_bytes) {
                if (T0 > 0) {
                    g.args[0].num_units = T0;
                    group_close(g, 1);
                    if (int st = launch<C>(kernel, g, num_sms, s)) return st;
                }
                GemmArgs& t = g.args[0];
                t.tile_begin = T0;
                t.num_units = R * split;
                t.split = split;
                t.kb_per = kb_per;
                t.partial_g = tail;
                group_close(g, 1);
                if (int st = launch<C>(kernel, g, num_sms, s)) return st;
                ReduceGroup<1> r;
                r.args[0] = t;
                r.count = 1;
                r.tile_m = C::TILE_M;
                r.tile_n = C::BN;
                r.block_begin[0] = 0;
                r.block_begin[1] = R * (C::TILE_M / 32) * (C::BN / 128);
                return launch_split_reduce<C>(r, s);
            }
        }
    }
    group_close(g, 1);
    return launch<C>(kernel, g, num_sms, s);
}

template <class C, class K>
int run_dw(K kernel, const uint16_t* X, const uint16_t* dY, const float* scale, const uint32_t* packed, float* gq,
           float* partial, int accumulate, float* tail, int64_t tail_bytes, int64_t M, int64_t K_, int64_t N,
           int num_sms, cudaStream_t s) {
    GemmGroup<1> g;
    GemmArgs a = make_args<C>(K_, N, M);
    a.out = gq;
    a.scale = scale;
    a.packed = packed;
    a.partial = partial;
    a.accumulate = accumulate;
    if (int st = group_set<C>(g, 0, X, K_, M, dY, nullptr, N, M, a)) return st;
    return dw_waves_and_tail<C>(kernel, g, tail, tail_bytes, kMaxTailUnits, num_sms, s);
}

}  // namespace

int gemm_status_read(int clear) {
    int v = 0;
    TERN_CUDA_TRY(cudaMemcpyFromSymbol(&v, g_gemm_status, sizeof(int)));
    if (clear) {
        const int zero[4] = {0, 0, 0, 0};
        TERN_CUDA_TRY(cudaMemcpyToSymbol(g_gemm_status, zero, sizeof(int)));
        TERN_CUDA_TRY(cudaMemcpyToSymbol(g_gemm_site, zero, sizeof(zero)));
    }
    return v ? TERN_ERR_TIMEOUT : TERN_OK;
}

}  // namespace tern

namespace tern {
int gemm_setup(int num_sms);   // every GEMM kernel configured once per device (below)
}  // namespace tern

using namespace tern;

extern "C" int tern_linear_fwd(const uint16_t* X, const tern_tiles* W, const float* scale, float* Y, int64_t M,
                               int64_t K, int64_t N, void* stream) {
    if (!X || !W || (!W->t_bf16 && !W->packed) || !scale || !Y) return TERN_ERR_ARG;
    if (!dims_ok(M, K, N)) return TERN_ERR_ARG;
    if (K % 16 || N % 16) return TERN_ERR_ALIGN;
    const void* b = W->t_bf16 ? static_cast<const void*>(W->t_bf16) : static_cast<const void*>(W->packed);
    if (!aligned16(X) || !aligned16(b) || !aligned16(scale) || !aligned16(Y)) return TERN_ERR_ALIGN;
    if (!W->t_bf16 && N % 64) return TERN_ERR_ALIGN;   // rows of 2-bit codes copied by TMA: 16-byte multiples
    int num_sms = 0;
    if (int st = check_device(&num_sms)) return st;
    if (int st = gemm_setup(num_sms)) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (W->t_bf16) {
        if (use_pair(M)) return run_fwd<Fwd2>(tern_fwd_gemm<2, 1>, X, W->t_bf16, nullptr, scale, Y, M, K, N, num_sms, s);
        return run_fwd<Fwd1>(tern_fwd_gemm<1, 1>, X, W->t_bf16, nullptr, scale, Y, M, K, N, num_sms, s);
    }
    if (use_pair(M)) return run_fwd<FwdP2>(tern_fwdp_gemm<2, 1>, X, nullptr, W->packed, scale, Y, M, K, N, num_sms, s);
    return run_fwd<FwdP1>(tern_fwdp_gemm<1, 1>, X, nullptr, W->packed, scale, Y, M, K, N, num_sms, s);
}

// sgrad partials: one row per 32-row group of K, rounded up to 256 bytes.
static int64_t bwd_partials_bytes(int64_t K, int64_t N) {
    const int64_t tiles_r = (K + kBM - 1) / kBM;
    return (tiles_r * 4 * N * static_cast<int64_t>(sizeof(float)) + 255) / 256 * 256;
}

extern "C" size_t tern_linear_bwd_workspace_min(int64_t M, int64_t K, int64_t N) {
    if (!dims_ok(M, K, N)) return 0;
    const int64_t tiles_r = (K + kBM - 1) / kBM;
    return static_cast<size_t>(tiles_r * 4 * N) * sizeof(float);
}

extern "C" size_t tern_linear_bwd_workspace(int64_t M, int64_t K, int64_t N) {
    if (!dims_ok(M, K, N)) return 0;
    const int64_t tail = use_pair(K) ? dw_tail_bytes<Dw2>(M, K, N) : dw_tail_bytes<Dw1>(M, K, N);
    return static_cast<size_t>(bwd_partials_bytes(K, N) + tail);
}

extern "C" size_t tern_linear_bwd_workspace_ex(int64_t M, int64_t K, int64_t N, unsigned flags) {
    if (!dims_ok(M, K, N) || (flags & ~static_cast<unsigned>(TERN_BWD_ACCUMULATE | TERN_BWD_DX_SPLIT8))) return 0;
    const size_t base = tern_linear_bwd_workspace(M, K, N);
    if (!(flags & TERN_BWD_DX_SPLIT8)) return base;
    return std::max(base, static_cast<size_t>(split8_dy_bytes(M, N)));
}

extern "C" int tern_linear_bwd_ex(const uint16_t* X, const uint16_t* dY, const tern_tiles* W, const float* scale,
                                  float* dX, float* gq, float* sgrad, void* workspace, size_t ws_bytes, int64_t M,
                                  int64_t K, int64_t N, unsigned flags, void* stream) {
    if (flags & ~static_cast<unsigned>(TERN_BWD_ACCUMULATE | TERN_BWD_DX_SPLIT8)) return TERN_ERR_ARG;
    const int accumulate = (flags & TERN_BWD_ACCUMULATE) ? 1 : 0;
    if (!X || !dY || !W || !scale) return TERN_ERR_ARG;
    const bool split8 = dX != nullptr && (flags & TERN_BWD_DX_SPLIT8) != 0;
    // without the hi/lo planes, dX expands them from the 2-bit codes inside the GEMM
    const bool codes = dX != nullptr && !split8 && !W->whi_bf16 && !W->wlo_bf16 && W->packed;
    if (dX && !split8 && !codes && (!W->whi_bf16 || !W->wlo_bf16)) return TERN_ERR_ARG;
    if (split8 && (!W->whi_f16 || !W->wlo_e4m3)) return TERN_ERR_ARG;
    if (sgrad && !W->packed) return TERN_ERR_ARG;
    if (!dX && !gq && !sgrad) return TERN_ERR_ARG;
    if (!dims_ok(M, K, N)) return TERN_ERR_ARG;
    if (K % 16 || N % 16) return TERN_ERR_ALIGN;
    if (!aligned16(X) || !aligned16(dY) || !aligned16(scale)) return TERN_ERR_ALIGN;
    if (sgrad && (!aligned16(sgrad) || !aligned16(W->packed) || !aligned16(workspace))) return TERN_ERR_ALIGN;
    if (gq && !aligned16(gq)) return TERN_ERR_ALIGN;
    if (dX && !split8 && !codes && (!aligned16(dX) || !aligned16(W->whi_bf16) || !aligned16(W->wlo_bf16)))
        return TERN_ERR_ALIGN;
    // the codes' rows are copied by TMA: N / 16 words a row, a 16-byte multiple
    if (codes && (!aligned16(dX) || !aligned16(W->packed) || N % 64 || (workspace && !aligned16(workspace))))
        return TERN_ERR_ALIGN;
    if (split8 && (!aligned16(dX) || !aligned16(W->whi_f16) || !aligned16(W->wlo_e4m3) ||
                   (workspace && !aligned16(workspace))))
        return TERN_ERR_ALIGN;
    if (sgrad && (!workspace || ws_bytes < tern_linear_bwd_workspace_min(M, K, N))) return TERN_ERR_WORKSPACE;
    if (split8 && (!workspace || static_cast<int64_t>(ws_bytes) < split8_dy_bytes(M, N))) return TERN_ERR_WORKSPACE;
    if (codes && (!workspace || static_cast<int64_t>(ws_bytes) < 4 * N)) return TERN_ERR_WORKSPACE;
    int num_sms = 0;
    if (int st = check_device(&num_sms)) return st;
    if (int st = gemm_setup(num_sms)) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    if (split8) {
        // dY's split into the workspace, read only by this dX GEMM (the G GEMM below
        // reuses the bytes after it on the same stream)
        uint16_t* dy16 = nullptr;
        uint8_t* dy8 = nullptr;
        int* rexp = nullptr;
        if (int st = split8_dy(dY, scale, M, N, workspace, &dy16, &dy8, &rexp, s)) return st;
        const int st = use_pair(M) ? run_dx8<Dx8_2>(tern_dx8_gemm<2, 1>, dy16, dy8, rexp, W->whi_f16, W->wlo_e4m3, dX,
                                                    M, K, N, num_sms, s)
                                   : run_dx8<Dx8_1>(tern_dx8_gemm<1, 1>, dy16, dy8, rexp, W->whi_f16, W->wlo_e4m3, dX,
                                                    M, K, N, num_sms, s);
        if (st) return st;
    } else if (codes) {
        // the s_hi / s_lo table into the workspace, read only by this dX GEMM (the G GEMM
        // below reuses the bytes after it on the same stream)
        uint16_t* hilo = static_cast<uint16_t*>(workspace);
        if (int st = scale_hilo(scale, N, hilo, s)) return st;
        const int st = use_pair(M) ? run_dxp<DxP2>(tern_dxp_gemm<2, 1>, dY, W->packed, hilo, dX, M, K, N, num_sms, s)
                                   : run_dxp<DxP1>(tern_dxp_gemm<1, 1>, dY, W->packed, hilo, dX, M, K, N, num_sms, s);
        if (st) return st;
    } else if (dX) {
        const int st = use_pair(M)
                           ? run_dx<Dx2>(tern_dx_gemm<2, 1>, dY, W->whi_bf16, W->wlo_bf16, dX, M, K, N, num_sms, s)
                           : run_dx<Dx1>(tern_dx_gemm<1, 1>, dY, W->whi_bf16, W->wlo_bf16, dX, M, K, N, num_sms, s);
        if (st) return st;
    }
    if (gq || sgrad) {
        float* partial = sgrad ? static_cast<float*>(workspace) : nullptr;
        // a workspace past the partials (16-byte aligned, 256-byte rounded) holds split G tiles
        const int64_t pb = sgrad ? bwd_partials_bytes(K, N) : 0;
        float* tail = nullptr;
        int64_t tail_bytes = 0;
        if (workspace && aligned16(workspace) && static_cast<int64_t>(ws_bytes) > pb) {
            tail = reinterpret_cast<float*>(static_cast<char*>(workspace) + pb);
            tail_bytes = static_cast<int64_t>(ws_bytes) - pb;
        }
        const int st = use_pair(K) ? run_dw<Dw2>(tern_dw_gemm<2, 1>, X, dY, scale, W->packed, gq, partial, accumulate,
                                                 tail, tail_bytes, M, K, N, num_sms, s)
                                   : run_dw<Dw1>(tern_dw_gemm<1, 1>, X, dY, scale, W->packed, gq, partial, accumulate,
                                                 tail, tail_bytes, M, K, N, num_sms, s);
        if (st) return st;
        if (!sgrad) return TERN_OK;
        const int nparts = static_cast<int>((K + kBM - 1) / kBM) * 4;
        if (int st = launch_pdl(tern_sgrad_reduce, dim3(static_cast<unsigned>((N + 255) / 256)), dim3(256), 0, s,
                                static_cast<const float*>(partial), nparts, static_cast<int>(N), sgrad, accumulate))
            return st;
    }
    return TERN_OK;
}

extern "C" int tern_linear_bwd(const uint16_t* X, const uint16_t* dY, const tern_tiles* W, const float* scale,
                               float* dX, float* gq, float* sgrad, void* workspace, size_t ws_bytes, int64_t M,
                               int64_t K, int64_t N, void* stream) {
    return tern_linear_bwd_ex(X, dY, W, scale, dX, gq, sgrad, workspace, ws_bytes, M, K, N, 0u, stream);
}

// ===================================================================== grouped calls
//
// Several independent layers per call (e.g. the projections of one block): up
// to kGroup problems share one persistent GEMM launch, so the tiles of small
// layers fill the GPU together and one layer's epilogue overlaps another's main
// loop.  Results equal the single-layer calls' up to the order of fp32 sums in
// the G tiles that are split along the token axis.

namespace tern {
namespace {


int layer_align(const tern_layer& L) {
    if (L.K % 16 || L.N % 16) return TERN_ERR_ALIGN;
    const void* ps[] = {L.X, L.dY, L.scale, L.Y, L.dX, L.gq, L.sgrad, L.Y_bf16, L.dX_bf16};
    for (const void* p : ps)
        if (p && !aligned16(p)) return TERN_ERR_ALIGN;
    const void* ws[] = {L.W->packed, L.W->t_bf16, L.W->whi_bf16, L.W->wlo_bf16};
    for (const void* p : ws)
        if (p && !aligned16(p)) return TERN_ERR_ALIGN;
    return TERN_OK;
}

// Calls fn(pair, idx, n) (or fn(pair, variant, idx, n)) for the layers selected by
// `pick`, in order, kGroup at a time, separately for layers whose rows (rows_of) need
// a CTA pair and those that do not, and for the two kernel variants `variant` tells
// apart (the forward's bf16 or 2-bit T).
template <class Pick, class Rows, class Var, class Fn>
int for_groups_v(const tern_layer* L, int count, Pick pick, Rows rows_of, Var variant, Fn fn) {
    for (int pair = 1; pair >= 0; --pair) {
        for (int v = 0; v < 2; ++v) {
            int idx[kGroup], n = 0;
            for (int i = 0; i <= count; ++i) {
                if (i < count && pick(L[i]) && use_pair(rows_of(L[i])) == (pair == 1) && variant(L[i]) == (v == 1))
                    idx[n++] = i;
                if (n == kGroup || (i == count && n > 0)) {
                    if (int st = fn(pair == 1, v == 1, idx, n)) return st;
                    n = 0;
                }
            }
        }
    }
    return TERN_OK;
}

template <class Pick, class Rows, class Fn>
int for_groups(const tern_layer* L, int count, Pick pick, Rows rows_of, Fn fn) {
    return for_groups_v(
        L, count, pick, rows_of, [](const tern_layer&) { return false; },
        [&](bool pair, bool, const int* idx, int n) { return fn(pair, idx, n); });
}

// The layers of a launch in descending order of k-blocks per tile (stable): the
// persistent pairs take units in concatenation order, so the longest tiles start
// first and the short ones fill the last wave.
template <class KbOf>
void longest_first(const int* idx, int n, int* out, KbOf kb_of) {
    for (int i = 0; i < n; ++i) out[i] = idx[i];
    std::stable_sort(out, out + n, [&](int a, int b) { return kb_of(a) > kb_of(b); });
}

template <class C, class K>
int fwd_group(K kernel, const tern_layer* L, const int* idx_in, int n, int num_sms, cudaStream_t s) {
    GemmGroup<kGroup> g;
    int idx[kGroup];
    longest_first(idx_in, n, idx, [&](int i) { return make_args<C>(L[i].M, L[i].N, L[i].K).num_kb; });
    for (int i = 0; i < n; ++i) {
        const tern_layer& l = L[idx[i]];
        GemmArgs a = make_args<C>(l.M, l.N, l.K);
        a.out = l.Y;
        a.out_bf16 = l.Y_bf16;
        a.scale = l.scale;
        a.bpacked = C::PK ? l.W->packed : nullptr;
        if (int st = group_set<C>(g, i, l.X, l.K, l.M, C::PK ? nullptr : l.W->t_bf16, nullptr, l.N, l.K, a))
            return st;
    }
    group_close(g, n);
    return launch<C>(kernel, g, num_sms, s);
}

template <class C, class K>
int dx_group(K kernel, const tern_layer* L, const int* idx_in, int n, int num_sms, cudaStream_t s) {
    GemmGroup<kGroup> g;
    int idx[kGroup];
    longest_first(idx_in, n, idx, [&](int i) { return make_args<C>(L[i].M, L[i].K, L[i].N).num_kb; });
    for (int i = 0; i < n; ++i) {
        const tern_layer& l = L[idx[i]];
        GemmArgs a = make_args<C>(l.M, l.K, l.N);
        a.out = l.dX;
        a.out_bf16 = l.dX_bf16;
        if (int st = group_set<C>(g, i, l.dY, l.N, l.M, l.W->whi_bf16, l.W->wlo_bf16, l.N, l.K, a)) return st;
    }
    group_close(g, n);
    return launch<C>(kernel, g, num_sms, s);
}

// Split factor for a group of G problems with `tiles` tiles in all: the one
// that minimises waves per slice, every problem keeping at least one k-block
// per slice and the split units within kMaxGroupTailUnits.
int group_split(int tiles, int min_kb, int units) {
    int best = 1;
    double best_cost = std::ceil(static_cast<double>(tiles) / units);
    for (int sp = 2; sp <= min_kb && tiles * sp <= kMaxGroupTailUnits; ++sp) {
        const double cost = std::ceil(static_cast<double>(tiles) * sp / units) / sp;
        if (cost < best_cost - 1e-9) {
            best = sp;
            best_cost = cost;
        }
    }
    return best;
}

template <class C>
int64_t group_tail_bytes(const tern_layer* L, const int* idx, int n) {
    int64_t units = 0;
    for (int i = 0; i < n; ++i) {
        const GemmArgs a = make_args<C>(L[idx[i]].K, L[idx[i]].N, L[idx[i]].M);
        units += static_cast<int64_t>(a.num_tiles) * a.num_kb;
    }
    return std::min<int64_t>(kMaxGroupTailUnits, units) * C::TILE_M * C::BN * static_cast<int64_t>(sizeof(float));
}

// The G GEMMs of a group with the fused gq / sgrad epilogue.  When the group's
// tiles leave persistent units idle and the workspace has room, every tile is
// split along the token axis by one factor and the grouped reduce finishes them.
template <class C, class K>
int dw_group(K kernel, const tern_layer* L, const int* idx, int n, float* const* partial, float* tail,
             int64_t tail_bytes, int accumulate, int num_sms, cudaStream_t s) {
    GemmGroup<kGroup> g;
    int pos[kGroup], order[kGroup];
    for (int i = 0; i < n; ++i) pos[i] = i;
    longest_first(pos, n, order, [&](int i) { return make_args<C>(L[idx[i]].K, L[idx[i]].N, L[idx[i]].M).num_kb; });
    int tiles = 0, min_kb = 1 << 30;
    for (int i = 0; i < n; ++i) {
        const tern_layer& l = L[idx[order[i]]];
        GemmArgs a = make_args<C>(l.K, l.N, l.M);
        a.out = l.gq;
        a.scale = l.scale;
        a.packed = l.W->packed;
        a.partial = partial[order[i]];
        a.accumulate = accumulate;
        if (int st = group_set<C>(g, i, l.X, l.K, l.M, l.dY, nullptr, l.N, l.M, a)) return st;
        tiles += a.num_tiles;
        min_kb = std::min(min_kb, a.num_kb);
    }
    int units = 0;
    if (int st = persistent_units<C>(kernel, num_sms, &units)) return st;
    int split = group_split(tiles, min_kb, units);
    const int64_t tile_bytes = static_cast<int64_t>(C::TILE_M) * C::BN * static_cast<int64_t>(sizeof(float));
    if (split >= 2 && static_cast<int64_t>(tiles) * split * tile_bytes > tail_bytes) split = 1;
    if (split == 1) {
        // one layer: whole waves, then its last wave's tiles split (as the single-layer call)
        if (n == 1) return dw_waves_and_tail<C>(kernel, g, tail, tail_bytes, kMaxGroupTailUnits, num_sms, s);
        group_close(g, n);
        return launch<C>(kernel, g, num_sms, s);
    }
    ReduceGroup<kGroup> r;
    r.count = n;
    r.tile_m = C::TILE_M;
    r.tile_n = C::BN;
    r.block_begin[0] = 0;
    int64_t off = 0;
    for (int i = 0; i < n; ++i) {
        GemmArgs& a = g.args[i];
        const int kb_per = (a.num_kb + split - 1) / split;
        a.split = (a.num_kb + kb_per - 1) / kb_per;   // every slice non-empty
        a.kb_per = kb_per;
        a.num_units = a.num_tiles * a.split;
        a.partial_g = tail + off;
        off += static_cast<int64_t>(a.num_units) * C::TILE_M * C::BN;
        r.args[i] = a;
        r.block_begin[i + 1] = r.block_begin[i] + a.num_tiles * (C::TILE_M / 32) * (C::BN / 128);
    }
    group_close(g, n);
    if (int st = launch<C>(kernel, g, num_sms, s)) return st;
    return launch_split_reduce<C>(r, s);
}

// sgrad of up to kGroup layers: each column sums its layer's partial rows in order.
struct SgradGroup {
    const float* partial[kGroup];
    float* sgrad[kGroup];
    int nparts[kGroup], N[kGroup];
    int block_begin[kGroup + 1];
    int count, accumulate;
};

}  // namespace

__global__ void __launch_bounds__(256) tern_sgrad_reduce_group(const __grid_constant__ SgradGroup g) {
    ptx::pdl_trigger();
    ptx::pdl_wait();
    int p = 0;
    while (p + 1 < g.count && static_cast<int>(blockIdx.x) >= g.block_begin[p + 1]) ++p;
    const int c = (static_cast<int>(blockIdx.x) - g.block_begin[p]) * blockDim.x + threadIdx.x;
    if (c >= g.N[p]) return;
    const float s = ordered_column_sum(g.partial[p], g.nparts[p], g.N[p], c);
    g.sgrad[p][c] = g.accumulate ? g.sgrad[p][c] + s : s;
}

}  // namespace tern

extern "C" int tern_linear_fwd_grouped(const tern_layer* layers, int count, void* stream) {
    if (!layers || count < 1) return TERN_ERR_ARG;
    for (int i = 0; i < count; ++i) {
        const tern_layer& l = layers[i];
        if (!l.X || !l.W || (!l.W->t_bf16 && !l.W->packed) || !l.scale || (!l.Y && !l.Y_bf16) ||
            !dims_ok(l.M, l.K, l.N))
            return TERN_ERR_ARG;
        if (int st = layer_align(l)) return st;
        if (!l.W->t_bf16 && l.N % 64) return TERN_ERR_ALIGN;
    }
    int num_sms = 0;
    if (int st = check_device(&num_sms)) return st;
    if (int st = gemm_setup(num_sms)) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return for_groups_v(
        layers, count, [](const tern_layer&) { return true; }, [](const tern_layer& l) { return l.M; },
        [](const tern_layer& l) { return l.W->t_bf16 == nullptr; },
        [&](bool pair, bool packed, const int* idx, int n) {
            if (packed)
                return pair ? fwd_group<FwdP2>(tern_fwdp_gemm<2, kGroup>, layers, idx, n, num_sms, s)
                            : fwd_group<FwdP1>(tern_fwdp_gemm<1, kGroup>, layers, idx, n, num_sms, s);
            return pair ? fwd_group<Fwd2>(tern_fwd_gemm<2, kGroup>, layers, idx, n, num_sms, s)
                        : fwd_group<Fwd1>(tern_fwd_gemm<1, kGroup>, layers, idx, n, num_sms, s);
        });
}

// Workspace of a grouped backward: every layer's sgrad partials (256-byte
// rounded, in layer order), then room for the split G tiles of the largest group.
extern "C" size_t tern_linear_bwd_grouped_workspace(const tern_layer* layers, int count) {
    if (!layers || count < 1) return 0;
    int64_t bytes = 0, tail = 0;
    for (int i = 0; i < count; ++i) {
        if (!dims_ok(layers[i].M, layers[i].K, layers[i].N)) return 0;
        bytes += bwd_partials_bytes(layers[i].K, layers[i].N);
    }
    for_groups(
        layers, count, [](const tern_layer&) { return true; }, [](const tern_layer& l) { return l.K; },
        [&](bool pair, const int* idx, int n) {
            tail = std::max(tail, pair ? group_tail_bytes<Dw2>(layers, idx, n) : group_tail_bytes<Dw1>(layers, idx, n));
            return TERN_OK;
        });
    return static_cast<size_t>(bytes + tail);
}

extern "C" int tern_linear_bwd_grouped(const tern_layer* layers, int count, void* workspace, size_t ws_bytes,
                                       unsigned flags, void* stream) {
    if (!layers || count < 1) return TERN_ERR_ARG;
    if (flags & ~static_cast<unsigned>(TERN_BWD_ACCUMULATE)) return TERN_ERR_ARG;
    const int accumulate = (flags & TERN_BWD_ACCUMULATE) ? 1 : 0;
    int64_t need = 0;
    for (int i = 0; i < count; ++i) {
        const tern_layer& l = layers[i];
        const bool dx = l.dX != nullptr || l.dX_bf16 != nullptr;
        if (!l.X || !l.dY || !l.W || !l.scale || (!dx && !l.gq && !l.sgrad)) return TERN_ERR_ARG;
        if (dx && (!l.W->whi_bf16 || !l.W->wlo_bf16)) return TERN_ERR_ARG;
        if (l.sgrad && !l.W->packed) return TERN_ERR_ARG;
        if (!dims_ok(l.M, l.K, l.N)) return TERN_ERR_ARG;
        if (int st = layer_align(l)) return st;
        need += bwd_partials_bytes(l.K, l.N);
    }
    if (!workspace) return TERN_ERR_WORKSPACE;
    if (!aligned16(workspace)) return TERN_ERR_ALIGN;
    if (static_cast<int64_t>(ws_bytes) < need) return TERN_ERR_WORKSPACE;
    int num_sms = 0;
    if (int st = check_device(&num_sms)) return st;
    if (int st = gemm_setup(num_sms)) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* ws = static_cast<char*>(workspace);
    float* tail = reinterpret_cast<float*>(ws + need);
    const int64_t tail_bytes = static_cast<int64_t>(ws_bytes) - need;

    // dX of every layer that asks for it
    if (int st = for_groups(
            layers, count, [](const tern_layer& l) { return l.dX != nullptr || l.dX_bf16 != nullptr; },
            [](const tern_layer& l) { return l.M; },
            [&](bool pair, const int* idx, int n) {
                return pair ? dx_group<Dx2>(tern_dx_gemm<2, kGroup>, layers, idx, n, num_sms, s)
                            : dx_group<Dx1>(tern_dx_gemm<1, kGroup>, layers, idx, n, num_sms, s);
            }))
        return st;

    // G with the fused gq / sgrad epilogue
    std::vector<float*> partial(count, nullptr);
    int64_t off = 0;
    for (int i = 0; i < count; ++i) {
        if (layers[i].sgrad) partial[i] = reinterpret_cast<float*>(ws + off);
        off += bwd_partials_bytes(layers[i].K, layers[i].N);
    }
    if (int st = for_groups(
            layers, count, [](const tern_layer& l) { return l.gq != nullptr || l.sgrad != nullptr; },
            [](const tern_layer& l) { return l.K; },
            [&](bool pair, const int* idx, int n) {
                float* parts[kGroup];
                for (int k = 0; k < n; ++k) parts[k] = partial[idx[k]];
                return pair ? dw_group<Dw2>(tern_dw_gemm<2, kGroup>, layers, idx, n, parts, tail, tail_bytes,
                                            accumulate, num_sms, s)
                            : dw_group<Dw1>(tern_dw_gemm<1, kGroup>, layers, idx, n, parts, tail, tail_bytes,
                                            accumulate, num_sms, s);
            }))
        return st;

    // sgrad sums
    SgradGroup sg{};
    sg.accumulate = accumulate;
    int n = 0;
    for (int i = 0; i <= count; ++i) {
        if (i < count && layers[i].sgrad) {
            sg.partial[n] = partial[i];
            sg.sgrad[n] = layers[i].sgrad;
            sg.nparts[n] = static_cast<int>((layers[i].K + kBM - 1) / kBM) * 4;
            sg.N[n] = static_cast<int>(layers[i].N);
            sg.block_begin[n + 1] = sg.block_begin[n] + static_cast<int>((layers[i].N + 255) / 256);
            ++n;
        }
        if (n == kGroup || (i == count && n > 0)) {
            sg.count = n;
            if (int st = launch_pdl(tern_sgrad_reduce_group, dim3(static_cast<unsigned>(sg.block_begin[n])),
                                    dim3(256), 0, s, sg))
                return st;
            n = 0;
        }
    }
    return TERN_OK;
}

namespace tern {

// Configure and load every GEMM kernel of the library once per device, before its
// first launch: the shared-memory attribute, the co-resident cluster count and the
// kernels' code (cudaFuncGetAttributes loads a lazily loaded kernel).  No kernel is
// then first used in the middle of a chain of dependent launches or under capture.
int gemm_setup(int num_sms) {
    static std::once_flag once[64];
    static int status[64];
    int dev = 0;
    TERN_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return TERN_ERR_DEVICE;
    std::call_once(once[dev], [&] {
        int st = TERN_OK, u = 0;
        auto gemm = [&](int r) {
            if (st == TERN_OK) st = r;
        };
        gemm(persistent_units<Fwd1>(tern_fwd_gemm<1, 1>, num_sms, &u));
        gemm(persistent_units<Fwd2>(tern_fwd_gemm<2, 1>, num_sms, &u));
        gemm(persistent_units<Dx1>(tern_dx_gemm<1, 1>, num_sms, &u));
        gemm(persistent_units<Dx2>(tern_dx_gemm<2, 1>, num_sms, &u));
        gemm(persistent_units<Dw1>(tern_dw_gemm<1, 1>, num_sms, &u));
        gemm(persistent_units<Dw2>(tern_dw_gemm<2, 1>, num_sms, &u));
        gemm(persistent_units<Fwd1>(tern_fwd_gemm<1, kGroup>, num_sms, &u));
        gemm(persistent_units<Fwd2>(tern_fwd_gemm<2, kGroup>, num_sms, &u));
        gemm(persistent_units<Dx1>(tern_dx_gemm<1, kGroup>, num_sms, &u));
        gemm(persistent_units<Dx2>(tern_dx_gemm<2, kGroup>, num_sms, &u));
        gemm(persistent_units<Dw1>(tern_dw_gemm<1, kGroup>, num_sms, &u));
        gemm(persistent_units<Dw2>(tern_dw_gemm<2, kGroup>, num_sms, &u));
        gemm(persistent_units<FwdP1>(tern_fwdp_gemm<1, 1>, num_sms, &u));
        gemm(persistent_units<FwdP2>(tern_fwdp_gemm<2, 1>, num_sms, &u));
        gemm(persistent_units<FwdP1>(tern_fwdp_gemm<1, kGroup>, num_sms, &u));
        gemm(persistent_units<FwdP2>(tern_fwdp_gemm<2, kGroup>, num_sms, &u));
        gemm(persistent_units<Dx8_1>(tern_dx8_gemm<1, 1>, num_sms, &u));
        gemm(persistent_units<DxP1>(tern_dxp_gemm<1, 1>, num_sms, &u));
        gemm(persistent_units<DxP2>(tern_dxp_gemm<2, 1>, num_sms, &u));
        gemm(persistent_units<Dx8_2>(tern_dx8_gemm<2, 1>, num_sms, &u));
        cudaFuncAttributes fa;
        auto load = [&](cudaError_t e) {
            if (st == TERN_OK && e != cudaSuccess) st = TERN_ERR_CUDA;
        };
        load(cudaFuncGetAttributes(&fa, tern_dw_split_reduce<1>));
        load(cudaFuncGetAttributes(&fa, tern_dw_split_reduce<kGroup>));
        load(cudaFuncGetAttributes(&fa, tern_sgrad_reduce));
        load(cudaFuncGetAttributes(&fa, tern_sgrad_reduce_group));
        status[dev] = st;
    });
    return status[dev];
}

}  // namespace tern

// ===================================================================== backward without a workspace
//
// tern_linear_bwd needs a device workspace for the sgrad partials, which the
// caller allocates.  Some callers cannot allocate device memory: a plugin run
// by a host program that owns every device allocation and hands none to its
// plugins, or a loop that must never pay cudaMalloc's implicit device-wide
// synchronisation.  tern_linear_bwd_noalloc serves them with a fixed scratch
// array that lives in this library's device image: every GPU that loads the
// library holds TERN_NOALLOC_SCRATCH_BYTES of it until the process exits.
//
// The host cannot pass the array's name to a kernel (in host code it is only a
// host-side stand-in for the symbol), so the first call on each device looks up
// its device address with cudaGetSymbolAddress while that device is current,
// and later calls on that device reuse it.  Make that first call on each device
// before any stream capture.
//
// Every call shares the one array and leaves its last contents behind.  Nothing
// needs clearing: the G kernel writes every partial the reduction reads.  Two
// calls whose kernels overlap on a GPU (different streams, no ordering between
// them) race on the array and give wrong sgrad values.

namespace tern {

static __device__ __align__(256) float g_noalloc_partials[TERN_NOALLOC_SCRATCH_BYTES / sizeof(float)];

namespace {

struct NoallocScratch {
    std::once_flag once;
    cudaError_t err = cudaErrorUnknown;
    void* ptr = nullptr;
};
NoallocScratch g_noalloc_scratch[64];

// Device address of g_noalloc_partials on the current device (set up once per device).
int noalloc_scratch(void** out) {
    int dev = 0;
    TERN_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return TERN_ERR_DEVICE;
    NoallocScratch& s = g_noalloc_scratch[dev];
    std::call_once(s.once, [&s] { s.err = cudaGetSymbolAddress(&s.ptr, g_noalloc_partials); });
    if (s.err != cudaSuccess || s.ptr == nullptr) return TERN_ERR_CUDA;
    *out = s.ptr;
    return TERN_OK;
}

}  // namespace
}  // namespace tern

extern "C" int tern_linear_bwd_noalloc(const uint16_t* X, const uint16_t* dY, const tern_tiles* W,
                                       const float* scale, float* dX, float* gq, float* sgrad, int64_t M,
                                       int64_t K, int64_t N, void* stream) {
    if (sgrad && tern_linear_bwd_workspace_min(M, K, N) > TERN_NOALLOC_SCRATCH_BYTES) return TERN_ERR_SCRATCH_LIMIT;
    void* scratch = nullptr;
    if (int st = noalloc_scratch(&scratch)) return st;
    return tern_linear_bwd(X, dY, W, scale, dX, gq, sgrad, scratch, TERN_NOALLOC_SCRATCH_BYTES, M, K, N, stream);
}

// ===================================================================== diagnostics
//
// Read while other streams may be stuck: the copy runs on the library's own
// non-blocking stream into pinned host memory (both created by the first call,
// which should therefore come while the device is healthy), and the host polls
// for at most `wait_ms`.

namespace tern {
namespace {

struct DiagState {
    std::once_flag once;
    cudaError_t err = cudaErrorUnknown;
    cudaStream_t stream = nullptr;
    unsigned char* host = nullptr;   // pinned: status int at 0, counters at 8, site words at 32
};
DiagState g_diag[64];

}  // namespace
}  // namespace tern

extern "C" int tern_device_diagnostics(int64_t* out, int wait_ms) {
    if (!out || wait_ms < 0) return TERN_ERR_ARG;
    int dev = 0;
    TERN_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return TERN_ERR_DEVICE;
    DiagState& d = g_diag[dev];
    std::call_once(d.once, [&d] {
        d.err = cudaStreamCreateWithFlags(&d.stream, cudaStreamNonBlocking);
        if (d.err == cudaSuccess) d.err = cudaHostAlloc(reinterpret_cast<void**>(&d.host), 64, cudaHostAllocDefault);
    });
    TERN_CUDA_TRY(d.err);
    // copy-engine reads: they do not need a free SM
    TERN_CUDA_TRY(cudaMemcpyFromSymbolAsync(d.host, g_gemm_status, sizeof(int), 0, cudaMemcpyDeviceToHost, d.stream));
    TERN_CUDA_TRY(cudaMemcpyFromSymbolAsync(d.host + 8, g_gemm_count, sizeof(g_gemm_count), 0,
                                            cudaMemcpyDeviceToHost, d.stream));
    TERN_CUDA_TRY(cudaMemcpyFromSymbolAsync(d.host + 32, g_gemm_site, sizeof(g_gemm_site), 0,
                                            cudaMemcpyDeviceToHost, d.stream));
    for (int t = 0; t <= wait_ms; ++t) {
        const cudaError_t q = cudaStreamQuery(d.stream);
        if (q == cudaSuccess) {
            int st = 0, site[4];
            unsigned long long cnt[3];
            std::memcpy(&st, d.host, sizeof(int));
            std::memcpy(cnt, d.host + 8, sizeof(cnt));
            std::memcpy(site, d.host + 32, sizeof(site));
            out[0] = st;
            for (int i = 0; i < 3; ++i) out[1 + i] = static_cast<int64_t>(cnt[i]);
            for (int i = 0; i < 4; ++i) out[4 + i] = site[i];
            return TERN_OK;
        }
        if (q != cudaErrorNotReady) return TERN_ERR_CUDA;
        std::this_thread::sleep_for(std::chrono::milliseconds(1));
    }
    return TERN_ERR_TIMEOUT;
}

extern "C" int tern_selftest_wait_timeout(unsigned limit_us, void* stream) {
    if (limit_us < 1 || limit_us > 2000000) return TERN_ERR_ARG;
    int num_sms = 0;
    if (int st = check_device(&num_sms)) return st;
    return launch_pdl(tern_wait_selftest, dim3(1), dim3(32), 0, static_cast<cudaStream_t>(stream),
                      static_cast<uint64_t>(limit_us) * 1000ull);
}
