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
// The kernel is HBM-bound: each thread owns one 16-element group (one packed
// word) per iteration, loads it as one 16-byte vector and stores every output
// with 16-byte (or 4-byte for packed) coalesced accesses.
#include <cuda_bf16.h>

#include "common.cuh"

namespace tern {

namespace {

struct MatArgs {
    const int8_t* q;
    int8_t* qc;
    const float* scale;
    uint32_t* packed;
    uint16_t* t;
    uint16_t* whi;
    uint16_t* wlo;
    int64_t groups;      // K * N / 16
    uint32_t ngroups_row;  // N / 16
    int theta, clamp;
};

__device__ __forceinline__ uint32_t bf16_bits(float x) {
    return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(x)));
}

}  // namespace

__global__ void __launch_bounds__(256) tern_materialize_kernel(const MatArgs a) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t gi = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; gi < a.groups; gi += stride) {
        const int64_t e0 = gi * 16;
        const int4 raw = __ldcs(reinterpret_cast<const int4*>(a.q + e0));
        const uint32_t words[4] = {static_cast<uint32_t>(raw.x), static_cast<uint32_t>(raw.y),
                                   static_cast<uint32_t>(raw.z), static_cast<uint32_t>(raw.w)};
        int w[16];
        uint32_t qcw[4] = {0, 0, 0, 0};
        uint32_t code = 0;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            int v = static_cast<int8_t>((words[j >> 2] >> (8 * (j & 3))) & 0xFFu);
            v = v > a.clamp ? a.clamp : (v < -a.clamp ? -a.clamp : v);
            qcw[j >> 2] |= (static_cast<uint32_t>(v) & 0xFFu) << (8 * (j & 3));
            w[j] = v >= a.theta ? 1 : (v <= -a.theta ? -1 : 0);
            code |= (w[j] == 1 ? 1u : (w[j] == -1 ? 3u : 0u)) << (2 * j);
        }
        if (a.qc) __stcs(reinterpret_cast<int4*>(a.qc + e0), make_int4(qcw[0], qcw[1], qcw[2], qcw[3]));
        if (a.packed) __stcs(a.packed + gi, code);
        if (a.t) {
            uint32_t p[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t lo = w[2 * i] == 0 ? 0u : (w[2 * i] > 0 ? 0x3F80u : 0xBF80u);
                const uint32_t hi = w[2 * i + 1] == 0 ? 0u : (w[2 * i + 1] > 0 ? 0x3F80u : 0xBF80u);
                p[i] = lo | (hi << 16);
            }
            int4* dst = reinterpret_cast<int4*>(a.t + e0);
            __stcs(dst, make_int4(p[0], p[1], p[2], p[3]));
            __stcs(dst + 1, make_int4(p[4], p[5], p[6], p[7]));
        }
        if (a.whi || a.wlo) {
            const uint32_t cg = static_cast<uint32_t>(gi % a.ngroups_row);
            const float4* sp = reinterpret_cast<const float4*>(a.scale + static_cast<int64_t>(cg) * 16);
            uint32_t hi_b[16], lo_b[16];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 s4 = __ldg(sp + i);
                const float s[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t hb = bf16_bits(s[k]);
                    const float hv = __uint_as_float(hb << 16);
                    hi_b[4 * i + k] = hb;
                    lo_b[4 * i + k] = bf16_bits(s[k] - hv);   // exact difference in fp32
                }
            }
            uint32_t ph[8], pl[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                uint32_t h2[2], l2[2];
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int j = 2 * i + k;
                    const uint32_t neg = w[j] < 0 ? 0x8000u : 0u;
                    h2[k] = w[j] == 0 ? 0u : (hi_b[j] ^ neg);
                    l2[k] = w[j] == 0 ? 0u : (lo_b[j] ^ neg);
                }
                ph[i] = h2[0] | (h2[1] << 16);
                pl[i] = l2[0] | (l2[1] << 16);
            }
            if (a.whi) {
                int4* dst = reinterpret_cast<int4*>(a.whi + e0);
                __stcs(dst, make_int4(ph[0], ph[1], ph[2], ph[3]));
                __stcs(dst + 1, make_int4(ph[4], ph[5], ph[6], ph[7]));
            }
            if (a.wlo) {
                int4* dst = reinterpret_cast<int4*>(a.wlo + e0);
                __stcs(dst, make_int4(pl[0], pl[1], pl[2], pl[3]));
                __stcs(dst + 1, make_int4(pl[4], pl[5], pl[6], pl[7]));
            }
        }
    }
}

}  // namespace tern

using namespace tern;

extern "C" int tern_materialize(const int8_t* q, int8_t* q_clamped, const float* scale, int64_t K, int64_t N,
                                int theta, int q_clamp, const tern_tiles* out, void* stream) {
    if (!q || !out) return TERN_ERR_ARG;
    if (K < 1 || N < 16 || K >= (1ll << 31) || N >= (1ll << 31) || K * N >= (1ll << 40)) return TERN_ERR_ARG;
    if (theta < 1 || q_clamp < theta || q_clamp > 127) return TERN_ERR_ARG;
    if ((out->whi_bf16 || out->wlo_bf16) && !scale) return TERN_ERR_ARG;
    if (N % 16) return TERN_ERR_ALIGN;
    const void* ptrs[] = {q, q_clamped, scale, out->packed, out->t_bf16, out->whi_bf16, out->wlo_bf16};
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
    a.theta = theta;
    a.clamp = q_clamp;
    const int64_t want = (a.groups + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
    tern_materialize_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(a);
    TERN_CUDA_TRY(cudaGetLastError());
    return TERN_OK;
}

extern "C" size_t tern_tiles_bytes(int64_t K, int64_t N, int which) {
    if (K < 1 || N < 16 || N % 16) return 0;
    switch (which) {
    case TERN_TILE_PACKED: return static_cast<size_t>(K * (N / 16)) * 4;
    case TERN_TILE_T:
    case TERN_TILE_WHI:
    case TERN_TILE_WLO: return static_cast<size_t>(K * N) * 2;
    default: return 0;
    }
}
