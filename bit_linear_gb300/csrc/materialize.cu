// Ternarisation and tile encoding of one weight matrix (page "train_gpu.cu":
// tg_tern_from_q turns the int4 accumulator q into w = sign(q) when |q| >= theta,
// else 0; SR4_Q_CLAMP bounds q to +-7).  The page writes an fp32 ternary matrix
// and then an fp32 W_eff every step; here one streaming pass reads q once and
// writes only the encodings the GEMMs consume:
//   packed  2-bit codes, 16 per uint32 (0 -> 00, +1 -> 01, -1 -> 11), LSB first
//   t       bf16 of T (forward B operand)
//   whi/wlo bf16 of s_hi[c]*T and s_lo[c]*T, the two-term bf16 split of
//           scale[c]*T used by the dX GEMM (s_hi = bf16(scale), s_lo =
//           bf16(scale - s_hi)); a zero weight is +0 in every plane
//   qc      the clamped accumulator
// The kernel is HBM-bound.  Each thread issues eight loads before using any and
// works on four weights at a time with byte-SIMD compares.  Packed-only launches
// take 16-weight groups (one packed word, a 16-byte q load); launches that write
// the bf16 planes take 8-weight halves, so every plane store is one 16-byte
// store per thread and a warp covers 512 contiguous bytes.
#include <algorithm>
#include <vector>

#include <cuda_bf16.h>

#include "common.cuh"

namespace tern {

namespace {

struct MatArgs {
    const int8_t* q;     // q and qc may be the same buffer (in-place clamp)
    int8_t* qc;
    const float* __restrict__ scale;
    uint32_t* __restrict__ packed;
    uint16_t* __restrict__ t;
    uint16_t* __restrict__ whi;
    uint16_t* __restrict__ wlo;
    int64_t groups;        // K * N / 16
    uint32_t ngroups_row;  // N / 16
    uint32_t th_pos;       // theta in every byte
    uint32_t th_neg;       // -theta in every byte
    uint32_t cl_pos;       // clamp in every byte
    uint32_t cl_neg;       // -clamp in every byte
};

__device__ __forceinline__ uint32_t bf16_bits(float x) {
    return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(x)));
}

// Two weights' 16-bit lanes from byte masks (0xFF / 0x00) of bytes b and b+1.
__device__ __forceinline__ uint32_t lanes16(uint32_t bytemask, uint32_t sel) {
    return __byte_perm(bytemask, 0u, sel);
}

// Sixteen weights (one packed word) per thread and call, for the launches that write no
// bf16 plane (those take encode_half).
template <bool QC, bool PK, bool TT, bool HL>
__device__ __forceinline__ void encode_group(const MatArgs& a, int4 raw, int64_t gi) {
    static_assert(!TT && !HL, "the bf16 planes are written eight weights at a time (encode_half)");
    const uint32_t w[4] = {static_cast<uint32_t>(raw.x), static_cast<uint32_t>(raw.y),
                           static_cast<uint32_t>(raw.z), static_cast<uint32_t>(raw.w)};
    uint32_t pos[4], neg[4];
    uint32_t code = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        pos[k] = __vcmpges4(w[k], a.th_pos);   // 0xFF where q >= theta
        neg[k] = __vcmples4(w[k], a.th_neg);   // 0xFF where q <= -theta
        // per byte: +1 -> 01, -1 -> 11, 0 -> 00; then gather the four 2-bit codes
        uint32_t x = (pos[k] & 0x01010101u) | (neg[k] & 0x03030303u);
        x = (x | (x >> 6) | (x >> 12) | (x >> 18)) & 0xFFu;
        code |= x << (8 * k);
    }
    const int64_t e0 = gi * 16;
    if constexpr (QC) {
        int4 c;
        c.x = static_cast<int>(__vmaxs4(__vmins4(w[0], a.cl_pos), a.cl_neg));
        c.y = static_cast<int>(__vmaxs4(__vmins4(w[1], a.cl_pos), a.cl_neg));
        c.z = static_cast<int>(__vmaxs4(__vmins4(w[2], a.cl_pos), a.cl_neg));
        c.w = static_cast<int>(__vmaxs4(__vmins4(w[3], a.cl_pos), a.cl_neg));
        __stcs(reinterpret_cast<int4*>(a.qc + e0), c);
    }
    if constexpr (PK) __stcs(a.packed + gi, code);
}

// Eight weights (half a packed word) per thread and call, for the launches that
// write the bf16 planes: each plane then takes one 16-byte store per thread, so
// a warp's store covers 512 contiguous bytes; the codes go out as 16-bit halves.
// Plain write-back stores here (streaming stores measured 1.5% slower for this
// write-heavy mix).
template <bool QC, bool PK, bool TT, bool HL>
__device__ __forceinline__ void encode_half(const MatArgs& a, int2 raw, int64_t h) {
    const uint32_t w[2] = {static_cast<uint32_t>(raw.x), static_cast<uint32_t>(raw.y)};
    uint32_t pos[2], neg[2];
    uint32_t code = 0;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        pos[k] = __vcmpges4(w[k], a.th_pos);
        neg[k] = __vcmples4(w[k], a.th_neg);
        uint32_t x = (pos[k] & 0x01010101u) | (neg[k] & 0x03030303u);
        x = (x | (x >> 6) | (x >> 12) | (x >> 18)) & 0xFFu;
        code |= x << (8 * k);
    }
    const int64_t e0 = h * 8;
    if constexpr (QC) {
        int2 c;
        c.x = static_cast<int>(__vmaxs4(__vmins4(w[0], a.cl_pos), a.cl_neg));
        c.y = static_cast<int>(__vmaxs4(__vmins4(w[1], a.cl_pos), a.cl_neg));
        __stcs(reinterpret_cast<int2*>(a.qc + e0), c);
    }
    if constexpr (PK) reinterpret_cast<unsigned short*>(a.packed)[h] = static_cast<unsigned short>(code);
    uint32_t nz[4], ng[4];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        nz[2 * k] = lanes16(pos[k] | neg[k], 0x1100u);
        nz[2 * k + 1] = lanes16(pos[k] | neg[k], 0x3322u);
        ng[2 * k] = lanes16(neg[k], 0x1100u);
        ng[2 * k + 1] = lanes16(neg[k], 0x3322u);
    }
    if constexpr (TT) {
        uint32_t p[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) p[i] = (nz[i] & 0x3F803F80u) | (ng[i] & 0x80008000u);
        *reinterpret_cast<int4*>(a.t + e0) = make_int4(p[0], p[1], p[2], p[3]);
    }
    if constexpr (HL) {
        const uint32_t cg = static_cast<uint32_t>(h % (2 * static_cast<int64_t>(a.ngroups_row)));   // 8-column group
        const float4* sp = reinterpret_cast<const float4*>(a.scale + static_cast<int64_t>(cg) * 8);
        uint32_t hi2[4], lo2[4];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const float4 s4 = __ldg(sp + i);
            const float sv[4] = {s4.x, s4.y, s4.z, s4.w};
            uint32_t hb[4], lb[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                hb[k] = bf16_bits(sv[k]);
                lb[k] = bf16_bits(sv[k] - __uint_as_float(hb[k] << 16));   // exact difference in fp32
            }
            hi2[2 * i] = hb[0] | (hb[1] << 16);
            hi2[2 * i + 1] = hb[2] | (hb[3] << 16);
            lo2[2 * i] = lb[0] | (lb[1] << 16);
            lo2[2 * i + 1] = lb[2] | (lb[3] << 16);
        }
        // a zero weight is +0; a negative weight flips the sign bit of s_hi / s_lo
        if (a.whi) {
            uint32_t p[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) p[i] = (hi2[i] & nz[i]) ^ (ng[i] & 0x80008000u);
            *reinterpret_cast<int4*>(a.whi + e0) = make_int4(p[0], p[1], p[2], p[3]);
        }
        if (a.wlo) {
            uint32_t p[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) p[i] = (lo2[i] & nz[i]) ^ (ng[i] & 0x80008000u);
            *reinterpret_cast<int4*>(a.wlo + e0) = make_int4(p[0], p[1], p[2], p[3]);
        }
    }
}

}  // namespace

// One weight's pass: thread tid of nth walks the weight's items (grid-stride), eight
// loads in flight before their encodes.
template <bool QC, bool PK, bool TT, bool HL>
__device__ __forceinline__ void materialize_body(const MatArgs& a, int64_t tid, int64_t nth) {
    constexpr int U = 8;
    if constexpr (TT || HL) {
        const int64_t halves = a.groups * 2;
        const int2* q2 = reinterpret_cast<const int2*>(a.q);
        int64_t h = tid;
        for (; h + (U - 1) * nth < halves; h += U * nth) {
            int2 r[U];
#pragma unroll
            for (int j = 0; j < U; ++j) r[j] = __ldcs(q2 + h + j * nth);
#pragma unroll
            for (int j = 0; j < U; ++j) encode_half<QC, PK, TT, HL>(a, r[j], h + j * nth);
        }
        for (; h < halves; h += nth) encode_half<QC, PK, TT, HL>(a, __ldcs(q2 + h), h);
    } else {
        const int4* q4 = reinterpret_cast<const int4*>(a.q);
        int64_t gi = tid;
        for (; gi + (U - 1) * nth < a.groups; gi += U * nth) {
            int4 r[U];
#pragma unroll
            for (int j = 0; j < U; ++j) r[j] = __ldcs(q4 + gi + j * nth);
#pragma unroll
            for (int j = 0; j < U; ++j) encode_group<QC, PK, TT, HL>(a, r[j], gi + j * nth);
        }
        for (; gi < a.groups; gi += nth) encode_group<QC, PK, TT, HL>(a, __ldcs(q4 + gi), gi);
    }
}

// Weights of a grouped call that request the same encodings: job j owns the blocks
// [block_begin[j], block_begin[j+1]) of the launch.
constexpr int kMatGroup = 16;
struct MatGroup {
    MatArgs job[kMatGroup];
    int block_begin[kMatGroup + 1];
    int count;
};

// Which encodings a launch writes is a template choice, so the packed-only
// ternarisation carries no registers for the bf16 planes.
template <bool QC, bool PK, bool TT, bool HL>
__global__ void __launch_bounds__(256) tern_materialize_kernel(const MatArgs a) {
    ptx::pdl_trigger();
    ptx::pdl_wait();
    materialize_body<QC, PK, TT, HL>(a, static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x,
                                     static_cast<int64_t>(gridDim.x) * blockDim.x);
}

// Several weights in one launch, each on its own range of blocks.
template <bool QC, bool PK, bool TT, bool HL>
__global__ void __launch_bounds__(256) tern_materialize_group_kernel(const __grid_constant__ MatGroup g) {
    ptx::pdl_trigger();
    ptx::pdl_wait();
    int j = 0;
    while (j + 1 < g.count && static_cast<int>(blockIdx.x) >= g.block_begin[j + 1]) ++j;
    const int b = static_cast<int>(blockIdx.x) - g.block_begin[j];
    const int nb = g.block_begin[j + 1] - g.block_begin[j];
    materialize_body<QC, PK, TT, HL>(g.job[j], static_cast<int64_t>(b) * blockDim.x + threadIdx.x,
                                     static_cast<int64_t>(nb) * blockDim.x);
}

// s_hi[c] = bf16(scale[c]) and s_lo[c] = bf16(scale[c] - s_hi[c]) as two bf16 arrays
// (hilo[c], hilo[N + c]): the values the hi/lo planes carry, for the dX GEMM that expands
// them from the 2-bit codes.
__global__ void __launch_bounds__(256) tern_scale_hilo_kernel(const float* __restrict__ scale, int N,
                                                               uint16_t* __restrict__ hilo) {
    ptx::pdl_trigger();
    ptx::pdl_wait();
    const int c = static_cast<int>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (c >= N) return;
    const float sv = scale[c];
    const uint32_t hb = bf16_bits(sv);
    hilo[c] = static_cast<uint16_t>(hb);
    hilo[N + c] = static_cast<uint16_t>(bf16_bits(sv - __uint_as_float(hb << 16)));   // exact difference in fp32
}

namespace {

template <bool QC, bool PK, bool TT, bool HL>
int launch_materialize(const MatArgs& a, int num_sms, cudaStream_t s) {
    auto kernel = tern_materialize_kernel<QC, PK, TT, HL>;
    static int per_sm = 0;   // resident CTAs per SM (the grid strides over the rest); same on every GB300
    if (per_sm == 0) {
        int b = 0;
        TERN_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kernel, 256, 0));
        per_sm = b > 0 ? b : 1;
    }
    const int64_t items = (TT || HL) ? 2 * a.groups : a.groups;   // eight- or sixteen-weight items
    const int64_t want = (items + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms) * per_sm;
    const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
    return launch_pdl(kernel, dim3(grid), dim3(256), 0, s, a);
}

// A grouped launch: each job gets blocks in proportion to its items (about eight items per
// thread), within the resident-CTA budget of the GPU.
template <bool QC, bool PK, bool TT, bool HL>
int launch_materialize_group(MatGroup& g, int num_sms, cudaStream_t s) {
    auto kernel = tern_materialize_group_kernel<QC, PK, TT, HL>;
    static int per_sm = 0;
    if (per_sm == 0) {
        int b = 0;
        TERN_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kernel, 256, 0));
        per_sm = b > 0 ? b : 1;
    }
    const int64_t cap = static_cast<int64_t>(num_sms) * per_sm;
    int64_t want[kMatGroup], total = 0;
    for (int j = 0; j < g.count; ++j) {
        const int64_t items = (TT || HL) ? 2 * g.job[j].groups : g.job[j].groups;
        want[j] = (items + 256 * 8 - 1) / (256 * 8);
        total += want[j];
    }
    g.block_begin[0] = 0;
    for (int j = 0; j < g.count; ++j) {
        int64_t nb = total <= cap ? want[j] : std::max<int64_t>(1, want[j] * cap / total);
        g.block_begin[j + 1] = g.block_begin[j] + static_cast<int>(nb);
    }
    return launch_pdl(kernel, dim3(static_cast<unsigned>(g.block_begin[g.count])), dim3(256), 0, s, g);
}

template <int QCv, int PKv, int TTv, int HLv>
int launch_group_sig(MatGroup& g, int n, cudaStream_t s) {
    return launch_materialize_group<QCv != 0, PKv != 0, TTv != 0, HLv != 0>(g, n, s);
}

// signature bits: 8 = clamp write-back, 4 = packed, 2 = bf16 T, 1 = hi/lo planes
int launch_group_by_sig(int sig, MatGroup& g, int n, cudaStream_t s) {
    switch (sig) {
#define TERN_SIG(v) \
    case v: return launch_group_sig<(v >> 3) & 1, (v >> 2) & 1, (v >> 1) & 1, v & 1>(g, n, s);
        TERN_SIG(1) TERN_SIG(2) TERN_SIG(3) TERN_SIG(4) TERN_SIG(5) TERN_SIG(6) TERN_SIG(7) TERN_SIG(8)
        TERN_SIG(9) TERN_SIG(10) TERN_SIG(11) TERN_SIG(12) TERN_SIG(13) TERN_SIG(14) TERN_SIG(15)
#undef TERN_SIG
    default: return TERN_OK;
    }
}

template <bool QC, bool PK, bool TT>
int dispatch_hl(const MatArgs& a, bool hl, int n, cudaStream_t s) {
    return hl ? launch_materialize<QC, PK, TT, true>(a, n, s) : launch_materialize<QC, PK, TT, false>(a, n, s);
}
template <bool QC, bool PK>
int dispatch_t(const MatArgs& a, bool tt, bool hl, int n, cudaStream_t s) {
    return tt ? dispatch_hl<QC, PK, true>(a, hl, n, s) : dispatch_hl<QC, PK, false>(a, hl, n, s);
}
template <bool QC>
int dispatch_pk(const MatArgs& a, bool pk, bool tt, bool hl, int n, cudaStream_t s) {
    return pk ? dispatch_t<QC, true>(a, tt, hl, n, s) : dispatch_t<QC, false>(a, tt, hl, n, s);
}

}  // namespace

}  // namespace tern

using namespace tern;

namespace tern {
namespace {

// Checks one weight's arguments and fills its launch arguments; the encodings it asks for
// come back as signature bits (8 clamp, 4 packed, 2 bf16 T, 1 hi/lo; 0 = nothing).
int mat_args(const int8_t* q, int8_t* q_clamped, const float* scale, int64_t K, int64_t N, int theta, int q_clamp,
             const tern_tiles* out, MatArgs* a, int* sig) {
    if (!q || !out) return TERN_ERR_ARG;
    if (K < 1 || N < 16 || K >= (1ll << 31) || N >= (1ll << 31) || K * N >= (1ll << 40)) return TERN_ERR_ARG;
    if (theta < 1 || q_clamp < theta || q_clamp > 127) return TERN_ERR_ARG;
    if ((out->whi_bf16 || out->wlo_bf16 || out->whi_f16 || out->wlo_e4m3) && !scale) return TERN_ERR_ARG;
    if (N % 16) return TERN_ERR_ALIGN;
    const void* ptrs[] = {q,           q_clamped,    scale,         out->packed, out->t_bf16,
                          out->whi_bf16, out->wlo_bf16, out->whi_f16, out->wlo_e4m3};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return TERN_ERR_ALIGN;
    a->q = q;
    a->qc = q_clamped;
    a->scale = scale;
    a->packed = out->packed;
    a->t = out->t_bf16;
    a->whi = out->whi_bf16;
    a->wlo = out->wlo_bf16;
    a->groups = K * N / 16;
    a->ngroups_row = static_cast<uint32_t>(N / 16);
    const uint32_t tb = static_cast<uint8_t>(theta), tn = static_cast<uint8_t>(-theta);
    const uint32_t cb = static_cast<uint8_t>(q_clamp), cn = static_cast<uint8_t>(-q_clamp);
    a->th_pos = tb * 0x01010101u;
    a->th_neg = tn * 0x01010101u;
    a->cl_pos = cb * 0x01010101u;
    a->cl_neg = cn * 0x01010101u;
    *sig = (q_clamped ? 8 : 0) | (out->packed ? 4 : 0) | (out->t_bf16 ? 2 : 0) |
           ((out->whi_bf16 || out->wlo_bf16) ? 1 : 0);
    return TERN_OK;
}

}  // namespace
}  // namespace tern

extern "C" int tern_materialize_grouped(const tern_mat_layer* layers, int count, int theta, int q_clamp,
                                        void* stream) {
    if (!layers || count < 1) return TERN_ERR_ARG;
    std::vector<MatArgs> args(static_cast<size_t>(count));
    std::vector<int> sigs(static_cast<size_t>(count));
    for (int i = 0; i < count; ++i) {
        const tern_mat_layer& l = layers[i];
        if (int st = mat_args(l.q, l.q_clamped, l.scale, l.K, l.N, theta, q_clamp, l.out, &args[i], &sigs[i]))
            return st;
    }
    int num_sms = 0;
    if (int st = check_device(&num_sms)) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    for (int sig = 1; sig < 16; ++sig) {   // one launch per set of requested encodings (16 weights at a time)
        MatGroup g;
        g.count = 0;
        for (int i = 0; i <= count; ++i) {
            if (i < count && sigs[i] == sig) g.job[g.count++] = args[i];
            if (g.count == kMatGroup || (i == count && g.count > 0)) {
                if (int st = launch_group_by_sig(sig, g, num_sms, s)) return st;
                g.count = 0;
            }
        }
    }
    for (int i = 0; i < count; ++i) {   // the fp16 + e4m3 dX planes, weight by weight
        const tern_mat_layer& l = layers[i];
        if (l.out->whi_f16 || l.out->wlo_e4m3)
            if (int st = split8_planes(l.q, l.scale, l.K, l.N, theta, l.out->whi_f16, l.out->wlo_e4m3, num_sms, s))
                return st;
    }
    return TERN_OK;
}

extern "C" int tern_materialize(const int8_t* q, int8_t* q_clamped, const float* scale, int64_t K, int64_t N,
                                int theta, int q_clamp, const tern_tiles* out, void* stream) {
    if (!q || !out) return TERN_ERR_ARG;
    if (K < 1 || N < 16 || K >= (1ll << 31) || N >= (1ll << 31) || K * N >= (1ll << 40)) return TERN_ERR_ARG;
    if (theta < 1 || q_clamp < theta || q_clamp > 127) return TERN_ERR_ARG;
    const bool s8 = out->whi_f16 != nullptr || out->wlo_e4m3 != nullptr;
    if ((out->whi_bf16 || out->wlo_bf16 || s8) && !scale) return TERN_ERR_ARG;
    if (N % 16) return TERN_ERR_ALIGN;
    const void* ptrs[] = {q,           q_clamped,    scale,         out->packed, out->t_bf16,
                          out->whi_bf16, out->wlo_bf16, out->whi_f16, out->wlo_e4m3};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return TERN_ERR_ALIGN;
    int num_sms = 0;
    if (int st = check_device(&num_sms)) return st;
    MatArgs a;
    a.q = q;
    a.qc = q_clamped;
    a.scale = scale;
    a.packed = out->packed;
    a.t = out->t_bf16;
    a.whi = out->whi_bf16;
    a.wlo = out->wlo_bf16;
    a.groups = K * N / 16;
    a.ngroups_row = static_cast<uint32_t>(N / 16);
    const uint32_t tb = static_cast<uint8_t>(theta), tn = static_cast<uint8_t>(-theta);
    const uint32_t cb = static_cast<uint8_t>(q_clamp), cn = static_cast<uint8_t>(-q_clamp);
    a.th_pos = tb * 0x01010101u;
    a.th_neg = tn * 0x01010101u;
    a.cl_pos = cb * 0x01010101u;
    a.cl_neg = cn * 0x01010101u;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool qc = q_clamped != nullptr, pk = out->packed != nullptr, tt = out->t_bf16 != nullptr;
    const bool hl = out->whi_bf16 != nullptr || out->wlo_bf16 != nullptr;
    if (qc || pk || tt || hl) {
        if (int st = qc ? dispatch_pk<true>(a, pk, tt, hl, num_sms, s) : dispatch_pk<false>(a, pk, tt, hl, num_sms, s))
            return st;
    }
    // the fp16 + e4m3 dX planes: a pass of their own (ternary(clamp(q)) = ternary(q), so an
    // in-place clamp before it changes nothing)
    if (s8) return split8_planes(q, scale, K, N, theta, out->whi_f16, out->wlo_e4m3, num_sms, s);
    return TERN_OK;
}

namespace tern {
int scale_hilo(const float* scale, int64_t N, uint16_t* hilo, cudaStream_t s) {
    return launch_pdl(tern_scale_hilo_kernel, dim3(static_cast<unsigned>((N + 255) / 256)), dim3(256), 0, s, scale,
                      static_cast<int>(N), hilo);
}
}  // namespace tern

extern "C" size_t tern_tiles_bytes(int64_t K, int64_t N, int which) {
    if (K < 1 || N < 16 || N % 16) return 0;
    switch (which) {
    case TERN_TILE_PACKED: return static_cast<size_t>(K * (N / 16)) * 4;
    case TERN_TILE_T:
    case TERN_TILE_WHI:
    case TERN_TILE_WLO:
    case TERN_TILE_WHI16: return static_cast<size_t>(K * N) * 2;
    case TERN_TILE_WLO8: return static_cast<size_t>(K * N);
    default: return 0;
    }
}
