// Operands of the dX GEMM in the fp16 + e4m3 split (this library's encoding; the
// pages form W_eff = scale[c]*T in fp32 and multiply by it, page "train_gpu.cu",
// header comment "Optimizer split").
//
// dX[m][r] = sum_c dY[m][c] * scale[c] * T[r][c].  Write scale[c] = a_c * 2^e_c with
// e_c = floor(log2|scale[c]|), a_c in +-[1, 2), h_c = f16(a_c) and
// l_c = e4m3(2^7 (a_c - h_c)), so that a_c = h_c + 2^-7 l_c within 2^-15 |a_c|.  With a
// per-row exponent e_m of dY,
//   dX[m][r] = 2^e_m * ( sum_c dY16[m][c] * h_c T[r][c] + sum_c dY8[m][c] * l_c T[r][c] )
//   dY16[m][c] = f16 (dY[m][c] * 2^(e_c - e_m))        exact (bf16 values in fp16 range)
//   dY8[m][c]  = e4m3(dY[m][c] * 2^(e_c - e_m - 7))
// The first sum is a binary16 GEMM at the bf16 rate, the second an e4m3 GEMM at twice
// that rate, into one accumulator: 1.5 bf16 passes instead of the two of the bf16
// hi/lo split.  e_m puts the row's largest |dY[m][c]| * 2^e_c in [2^14, 2^15), so dY16
// stays below the binary16 limit and dY8 below 2^8 (e4m3's largest value is 448).
//
// This file holds the two encoding passes: the weight planes h_c T / l_c T (from q,
// with tern_materialize) and the per-call split of dY (with the dX GEMM).
#include <algorithm>
#include <climits>

#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"

namespace tern {
namespace {

__device__ __forceinline__ uint8_t e4m3_rn(float x) {
    return static_cast<uint8_t>(__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3));
}

// scale = a * 2^e with a in +-[1, 2): h = f16(a), l = e4m3(2^7 (a - h)); a zero scale
// gives h = l = 0.
__device__ __forceinline__ void column_split(float s, uint32_t& h, uint32_t& l) {
    const uint32_t u = __float_as_uint(s);
    uint32_t mag = u & 0x7FFFFFFFu;
    if (mag == 0) {
        h = 0;
        l = 0;
        return;
    }
    if (mag < 0x00800000u) mag <<= (__clz(mag) - 8);   // subnormal: bring the leading one to bit 23
    const float a = __uint_as_float((u & 0x80000000u) | 0x3F800000u | (mag & 0x007FFFFFu));
    const __half hh = __float2half_rn(a);
    h = __half_as_ushort(hh);
    l = e4m3_rn((a - __half2float(hh)) * 128.0f);   // the difference and the rescale are exact
}

// floor(log2|x|) of a nonzero finite fp32 value, normal or subnormal.
__device__ __forceinline__ int ilog2f(uint32_t bits) {
    const uint32_t a = bits & 0x7FFFFFFFu;
    const int ex = static_cast<int>(a >> 23);
    return ex ? ex - 127 : (31 - __clz(a)) - 149;
}

// x * 2^e for a finite fp32 x (bit pattern) whose result lies below 2^16: exact when the
// result is an fp32 normal, else (below 2^-126, where binary16 and e4m3 both round to
// zero) a signed zero.
__device__ __forceinline__ float scale_pow2(uint32_t u, int e) {
    const uint32_t sign = u & 0x80000000u;
    uint32_t a = u & 0x7FFFFFFFu;
    if (a == 0) return __uint_as_float(sign);
    int ex = static_cast<int>(a >> 23);
    if (ex == 0) {   // subnormal: normalise
        const int sh = __clz(a) - 8;
        a = (a << sh) & 0x007FFFFFu;
        ex = 1 - sh;
    } else {
        a &= 0x007FFFFFu;
    }
    const int ne = ex + e;
    if (ne <= 0) return __uint_as_float(sign);
    return __uint_as_float(sign | (static_cast<uint32_t>(ne) << 23) | a);
}

// ---------------------------------------------------------------- weight planes
//
// Thread t owns 16-column group t % G of every (t / G + i * rows_step)-th row, so the
// 16 column values h_c, l_c are computed once per thread; consecutive threads read
// consecutive 16-byte groups of a row of q.
__global__ void __launch_bounds__(256) tern_split8_planes_kernel(const int8_t* __restrict__ q,
                                                                  const float* __restrict__ scale, int64_t K,
                                                                  int groups_row, int rows_step, uint32_t th_pos,
                                                                  uint32_t th_neg, uint16_t* __restrict__ wh16,
                                                                  uint8_t* __restrict__ wl8) {
    ptx::pdl_trigger();
    ptx::pdl_wait();
    const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int cg = static_cast<int>(t % groups_row);
    int64_t r = t / groups_row;
    if (r >= rows_step) return;
    uint32_t h2[8], l4[4];   // the group's 16 h (two per word) and l (four per word)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float4 s4 = __ldg(reinterpret_cast<const float4*>(scale + static_cast<int64_t>(cg) * 16) + i);
        uint32_t h[4], l[4];
        column_split(s4.x, h[0], l[0]);
        column_split(s4.y, h[1], l[1]);
        column_split(s4.z, h[2], l[2]);
        column_split(s4.w, h[3], l[3]);
        h2[2 * i] = h[0] | (h[1] << 16);
        h2[2 * i + 1] = h[2] | (h[3] << 16);
        l4[i] = l[0] | (l[1] << 8) | (l[2] << 16) | (l[3] << 24);
    }
    const int64_t N = static_cast<int64_t>(groups_row) * 16;
    for (; r < K; r += rows_step) {
        const int64_t e0 = r * N + static_cast<int64_t>(cg) * 16;
        const int4 raw = __ldcs(reinterpret_cast<const int4*>(q + e0));
        const uint32_t w[4] = {static_cast<uint32_t>(raw.x), static_cast<uint32_t>(raw.y),
                               static_cast<uint32_t>(raw.z), static_cast<uint32_t>(raw.w)};
        uint32_t ph[8], pl[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t pos = __vcmpges4(w[k], th_pos);   // 0xFF where q >= theta
            const uint32_t neg = __vcmples4(w[k], th_neg);   // 0xFF where q <= -theta
            const uint32_t nz = pos | neg;
            // a zero weight is +0; a negative weight flips the sign bit
            pl[k] = (l4[k] & nz) ^ (neg & 0x80808080u);
            const uint32_t nz_lo = __byte_perm(nz, 0u, 0x1100u), nz_hi = __byte_perm(nz, 0u, 0x3322u);
            const uint32_t ng_lo = __byte_perm(neg, 0u, 0x1100u), ng_hi = __byte_perm(neg, 0u, 0x3322u);
            ph[2 * k] = (h2[2 * k] & nz_lo) ^ (ng_lo & 0x80008000u);
            ph[2 * k + 1] = (h2[2 * k + 1] & nz_hi) ^ (ng_hi & 0x80008000u);
        }
        if (wh16) {
            int4* d = reinterpret_cast<int4*>(wh16 + e0);
            d[0] = make_int4(ph[0], ph[1], ph[2], ph[3]);
            d[1] = make_int4(ph[4], ph[5], ph[6], ph[7]);
        }
        if (wl8) *reinterpret_cast<int4*>(wl8 + e0) = make_int4(pl[0], pl[1], pl[2], pl[3]);
    }
}

// ---------------------------------------------------------------- the split of dY
//
// The column factors 2^e_c first (0 for a zero scale) with the range of e_c, then one
// block per row of dY, eight columns (one 16-byte load) per chunk; up to kCh chunks per
// thread stay in registers between the block's two passes (the rest are read again).
// A row takes the fp32 path (a multiply per value, exact while the products are fp32
// normals) when its largest product and every column's 2^(e_c - e_m) are fp32 normals,
// else the integer path (exponent arithmetic on the bit patterns).
constexpr int kCh = 3;

// 2^e as fp32 for e in [-149, 127] (subnormal below -126).
__device__ __forceinline__ float pow2f(int e) {
    return e >= -126 ? __uint_as_float(static_cast<uint32_t>(e + 127) << 23) : __uint_as_float(1u << (e + 149));
}

__global__ void __launch_bounds__(1024) tern_split8_colexp_kernel(const float* __restrict__ scale, int N,
                                                                   float* __restrict__ fac, int* __restrict__ ext) {
    ptx::pdl_trigger();
    ptx::pdl_wait();
    __shared__ int rlo[32], rhi[32];
    int lo = INT_MAX, hi = INT_MIN;
    for (int c = static_cast<int>(threadIdx.x); c < N; c += static_cast<int>(blockDim.x)) {
        const uint32_t sb = __float_as_uint(scale[c]);
        float f = 0.0f;
        if (sb & 0x7FFFFFFFu) {
            const int e = ilog2f(sb);
            f = pow2f(e);
            lo = min(lo, e);
            hi = max(hi, e);
        }
        fac[c] = f;
    }
    lo = __reduce_min_sync(0xffffffffu, lo);
    hi = __reduce_max_sync(0xffffffffu, hi);
    if ((threadIdx.x & 31) == 0) {
        rlo[threadIdx.x >> 5] = lo;
        rhi[threadIdx.x >> 5] = hi;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int k = 1; k < static_cast<int>(blockDim.x >> 5); ++k) {
            lo = min(lo, rlo[k]);
            hi = max(hi, rhi[k]);
        }
        ext[0] = lo == INT_MAX ? 0 : lo;   // no nonzero scale: every output is zero
        ext[1] = hi == INT_MIN ? 0 : hi;
    }
}

__device__ __forceinline__ float bf16_at(const uint32_t (&w)[4], int j) {
    return __uint_as_float((j & 1) ? (w[j >> 1] & 0xFFFF0000u) : (w[j >> 1] << 16));
}

// Block-wide maximum of a non-negative int (or of non-negative fp32 bit patterns, which
// order like their values).
__device__ __forceinline__ int block_max(int v, int* red) {
    v = __reduce_max_sync(0xffffffffu, v);
    __syncthreads();   // red is reused
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    v = red[0];
    for (int k = 1; k < static_cast<int>(blockDim.x >> 5); ++k) v = max(v, red[k]);
    return v;
}

__global__ void __launch_bounds__(512, 3) tern_split8_dy_kernel(const uint16_t* __restrict__ dY,
                                                              const float* __restrict__ fac,
                                                              const int* __restrict__ ext, int N,
                                                              uint16_t* __restrict__ dy16, uint8_t* __restrict__ dy8,
                                                              int* __restrict__ row_exp) {
    ptx::pdl_trigger();
    ptx::pdl_wait();
    __shared__ int red[16];
    const int64_t row = blockIdx.x;
    const int chunks = N / 8, tid = static_cast<int>(threadIdx.x), nt = static_cast<int>(blockDim.x);
    const uint4* src = reinterpret_cast<const uint4*>(dY + row * N);
    const float4* facv = reinterpret_cast<const float4*>(fac);
    uint4 keep[kCh];
#pragma unroll
    for (int i = 0; i < kCh; ++i)
        if (tid + i * nt < chunks) keep[i] = __ldcs(src + tid + i * nt);
    auto factors = [&](int ch, float (&f)[8]) {
        const float4 f0 = __ldg(facv + 2 * ch), f1 = __ldg(facv + 2 * ch + 1);
        f[0] = f0.x, f[1] = f0.y, f[2] = f0.z, f[3] = f0.w, f[4] = f1.x, f[5] = f1.y, f[6] = f1.z, f[7] = f1.w;
    };
    // every chunk of the row once: the kCh kept ones, then the rest from global memory
    auto for_chunks = [&](auto&& fn) {
#pragma unroll
        for (int i = 0; i < kCh; ++i)
            if (tid + i * nt < chunks) fn(keep[i], tid + i * nt);
        for (int ch = tid + kCh * nt; ch < chunks; ch += nt) fn(__ldcs(src + ch), ch);
    };
    auto for_chunks_again = [&](auto&& fn) {   // the integer path (rare) reads the row again
        for (int ch = tid; ch < chunks; ch += nt) fn(__ldg(src + ch), ch);
    };
    auto store = [&](int ch, const float (&y)[8]) {
        uint32_t o16[4], o8[4];
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
            const __half2 hv = __floats2half2_rn(y[j], y[j + 1]);   // .x (low half) = column j
            o16[j >> 1] = *reinterpret_cast<const uint32_t*>(&hv);
            // the e4m3 copy is 2^-7 of the binary16 one (exact for fp32 normals; below 2^-126
            // both formats give zero)
            o8[j >> 1] = __nv_cvt_float2_to_fp8x2(make_float2(y[j] * 0.0078125f, y[j + 1] * 0.0078125f),
                                                 __NV_SATFINITE, __NV_E4M3);   // low byte = column j
        }
        reinterpret_cast<uint4*>(dy16 + row * N)[ch] = make_uint4(o16[0], o16[1], o16[2], o16[3]);
        reinterpret_cast<uint2*>(dy8 + row * N)[ch] = make_uint2(o8[0] | (o8[1] << 16), o8[2] | (o8[3] << 16));
    };

    // pass 1, fp32: the row's largest |dY[c]| * 2^e_c
    float mx = 0.0f;
    for_chunks([&](const uint4& v, int ch) {
        float f[8];
        factors(ch, f);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) mx = fmaxf(mx, fabsf(bf16_at(w, j)) * f[j]);
    });
    const uint32_t mb = static_cast<uint32_t>(block_max(static_cast<int>(__float_as_uint(mx)), red));
    int em = static_cast<int>(mb >> 23) - 127 - 14;
    const bool fast = mb >= 0x00800000u && mb < 0x7F800000u && em >= -126 && em <= 126 && ext[0] - em >= -126 &&
                      ext[1] - em <= 127;   // the same for the whole block
    if (fast) {
        // pass 2: y = dY[c] * (2^e_c * 2^-e_m), both factors and the product fp32 normals
        const float sm = pow2f(-em);
        for_chunks([&](const uint4& v, int ch) {
            float f[8], y[8];
            factors(ch, f);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 8; ++j) y[j] = bf16_at(w, j) * (f[j] * sm);
            store(ch, y);
        });
    } else {
        // the integer path: E = max of floor(log2|dY[c]|) + e_c over nonzero values and scales
        int E = INT_MIN;
        for_chunks_again([&](const uint4& v, int ch) {
            float f[8];
            factors(ch, f);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll 1
            for (int j = 0; j < 8; ++j) {
                const uint32_t b = __float_as_uint(bf16_at(w, j));
                if ((b & 0x7FFFFFFFu) && f[j] != 0.0f) E = max(E, ilog2f(b) + ilog2f(__float_as_uint(f[j])));
            }
        });
        E = block_max(E, red);
        em = E == INT_MIN ? 0 : E - 14;
        for_chunks_again([&](const uint4& v, int ch) {
            float f[8], y[8];
            factors(ch, f);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll 1
            for (int j = 0; j < 8; ++j)
                y[j] = f[j] == 0.0f ? 0.0f
                                    : scale_pow2(__float_as_uint(bf16_at(w, j)), ilog2f(__float_as_uint(f[j])) - em);
            store(ch, y);
        });
    }
    if (threadIdx.x == 0) row_exp[row] = em;
}

int64_t round256(int64_t b) { return (b + 255) / 256 * 256; }

}  // namespace

int split8_planes(const int8_t* q, const float* scale, int64_t K, int64_t N, int theta, uint16_t* wh16,
                  uint8_t* wl8, int num_sms, cudaStream_t s) {
    const int groups_row = static_cast<int>(N / 16);
    // rows per sweep: about 16 resident 256-thread blocks per SM in total
    const int64_t want_threads = static_cast<int64_t>(num_sms) * 16 * 256;
    const int64_t rows_step = std::max<int64_t>(1, std::min<int64_t>(K, want_threads / groups_row));
    const int64_t threads = rows_step * groups_row;
    const uint32_t tb = static_cast<uint8_t>(theta), tn = static_cast<uint8_t>(-theta);
    return launch_pdl(tern_split8_planes_kernel, dim3(static_cast<unsigned>((threads + 255) / 256)), dim3(256), 0, s,
                      q, scale, K, groups_row, static_cast<int>(rows_step), tb * 0x01010101u, tn * 0x01010101u, wh16,
                      wl8);
}

int64_t split8_dy_bytes(int64_t M, int64_t N) {
    return round256(M * N * 2) + round256(M * N) + round256(M * 4) + round256(N * 4) + 256;
}

int split8_dy(const uint16_t* dY, const float* scale, int64_t M, int64_t N, void* ws, uint16_t** dy16, uint8_t** dy8,
              int** row_exp, cudaStream_t s) {
    char* p = static_cast<char*>(ws);
    *dy16 = reinterpret_cast<uint16_t*>(p);
    p += round256(M * N * 2);
    *dy8 = reinterpret_cast<uint8_t*>(p);
    p += round256(M * N);
    *row_exp = reinterpret_cast<int*>(p);
    p += round256(M * 4);
    float* fac = reinterpret_cast<float*>(p);
    int* ext = reinterpret_cast<int*>(p + round256(N * 4));
    if (int st = launch_pdl(tern_split8_colexp_kernel, dim3(1), dim3(1024), 0, s, scale, static_cast<int>(N), fac, ext))
        return st;
    // threads per row: enough that each holds at most kCh chunks, one warp to sixteen
    const int64_t chunks = N / 8;
    int tpr = 32;
    while (tpr < 512 && chunks > kCh * tpr) tpr *= 2;
    return launch_pdl(tern_split8_dy_kernel, dim3(static_cast<unsigned>(M)), dim3(tpr), 0, s, dY,
                      static_cast<const float*>(fac), static_cast<const int*>(ext), static_cast<int>(N), *dy16, *dy8,
                      *row_exp);
}

}  // namespace tern
