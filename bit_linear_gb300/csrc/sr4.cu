// SR4 step: stochastic-rounding update of the int4 accumulator q from the
// straight-through gradient gq (page "train_gpu.cu": sr4_dev runs
// fc_sr4_scale<<<1,1>>> and then fc_sr4_update; the bodies are off the page).
// Reading implemented here (the same reading the oracle states):
//
//   s    = target_step / mean_i |gq_i * inv_bs|             (0 when the mean is 0)
//   q_i <- clamp(q_i - floor(x_i + u_i), +-q_clamp),  x_i = (gq_i * inv_bs) * s
//
// u_i ~ U[0,1) from a counter-based splitmix64 stream keyed by (seed, counter)
// and indexed by the global element index idx_base + i (u_i = 1/2 without
// dither); a non-finite x_i leaves q_i unchanged.
//
// Three launches instead of the page's single-thread scale kernel:
//   1. tern_sr4_absum     per-CTA sums of |gq*inv_bs| over fixed contiguous slices
//                         (deterministic): each thread keeps an fp32 sum and the
//                         exact error of its additions (two-sum), the CTA adds the
//                         threads' pairs in fp64; written to the workspace;
//   2. tern_sr4_finalize  one CTA: fixed-order sum, mean, s (fp32);
//   3. tern_sr4_update    streaming update, 16 weights per thread per iteration
//                         (16-byte q loads/stores, 4 float4 gq loads).
// The update's arithmetic uses explicitly rounded fp32 operations (no fused
// multiply-add), so the rounding decision is the oracle's decision.
#include "common.cuh"

namespace tern {

namespace {

constexpr int kAbsumBlocks = 1024;   // fixed slicing: the sum order does not depend on the GPU
constexpr uint64_t kG = 0x9E3779B97F4A7C15ull;

__host__ __device__ __forceinline__ uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

struct Sr4Args {
    int8_t* q;
    const float* gq;
    int64_t n;
    float inv_bs, target;
    uint64_t key;        // mix64(seed ^ counter*G)
    int64_t idx_base;
    int clamp, dither;
    double* partial;     // [kAbsumBlocks]
    float* s;            // device step scalar
    float* s_out;        // optional copy for the caller
};

// Counter of element i: key + (idx_base + i + 1) * G (mod 2^64); consecutive
// elements step by G.
__device__ __forceinline__ uint64_t sr4_counter(const Sr4Args& a, int64_t i) {
    return a.key + static_cast<uint64_t>(a.idx_base + i + 1) * kG;
}

// The top 24 bits of mix64(z): the final xor-shift by 31 does not reach bits
// 40..63, so they are bits 40..63 of the second product, whose upper 32 bits need
// one high and two low 32-bit multiplies instead of a full 64-bit product.
__device__ __forceinline__ uint32_t mix64_top24(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    const uint64_t y = z ^ (z >> 27);
    constexpr uint32_t c_lo = 0x133111EBu, c_hi = 0x94D049BBu;   // 0x94D049BB133111EB
    const uint32_t y_lo = static_cast<uint32_t>(y), y_hi = static_cast<uint32_t>(y >> 32);
    const uint32_t top = __umulhi(y_lo, c_lo) + y_lo * c_hi + y_hi * c_lo;   // bits 32..63 of y * c
    return top >> 8;
}

__device__ __forceinline__ int8_t sr4_one(const Sr4Args& a, int8_t q, float g, float s, uint64_t z) {
    const float x = __fmul_rn(__fmul_rn(g, a.inv_bs), s);
    float u = 0.5f;
    if (a.dither) u = static_cast<float>(mix64_top24(z)) * (1.0f / 16777216.0f);
    const float y = __fadd_rn(x, u);
    if (!isfinite(y)) return q;
    const float f = fminf(fmaxf(floorf(y), -300.0f), 300.0f);
    int v = static_cast<int>(q) - static_cast<int>(f);
    v = v > a.clamp ? a.clamp : (v < -a.clamp ? -a.clamp : v);
    return static_cast<int8_t>(v);
}

}  // namespace

// s + c += x as an unevaluated pair of fp32 values (Knuth's two-sum gives the
// rounding error of each addition exactly), so a thread's partial sum keeps about
// twice fp32's precision while the loop runs at fp32 rate.
__device__ __forceinline__ void two_sum_add(float& s, float& c, float x) {
    const float t = __fadd_rn(s, x);
    const float xv = __fsub_rn(t, s);
    const float sv = __fsub_rn(t, xv);
    const float e = __fadd_rn(__fsub_rn(s, sv), __fsub_rn(x, xv));
    s = t;
    c = __fadd_rn(c, e);
}

__global__ void __launch_bounds__(256) tern_sr4_absum(const Sr4Args a) {
    ptx::pdl_trigger();
    ptx::pdl_wait();
    // block b owns the float4 groups [b*n4/B, (b+1)*n4/B); the last block also the
    // n % 4 trailing elements.  Fixed slicing: the sum order does not depend on the GPU.
    const int64_t n4 = a.n / 4;
    const int64_t lo = n4 * blockIdx.x / gridDim.x, hi = n4 * (blockIdx.x + 1) / gridDim.x;
    const float4* g4 = reinterpret_cast<const float4*>(a.gq);
    float s = 0.0f, c = 0.0f;
#pragma unroll 4
    for (int64_t i = lo + threadIdx.x; i < hi; i += blockDim.x) {
        const float4 v = __ldg(g4 + i);
        two_sum_add(s, c, fabsf(__fmul_rn(v.x, a.inv_bs)));
        two_sum_add(s, c, fabsf(__fmul_rn(v.y, a.inv_bs)));
        two_sum_add(s, c, fabsf(__fmul_rn(v.z, a.inv_bs)));
        two_sum_add(s, c, fabsf(__fmul_rn(v.w, a.inv_bs)));
    }
    if (blockIdx.x == gridDim.x - 1) {
        const int64_t t = n4 * 4 + threadIdx.x;
        if (t < a.n) two_sum_add(s, c, fabsf(__fmul_rn(a.gq[t], a.inv_bs)));
    }
    __shared__ double red[256];
    red[threadIdx.x] = static_cast<double>(s) + static_cast<double>(c);
    __syncthreads();
    for (int w = 128; w > 0; w >>= 1) {
        if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) a.partial[blockIdx.x] = red[0];
}

__global__ void __launch_bounds__(256) tern_sr4_finalize(const Sr4Args a, int nparts) {
    ptx::pdl_trigger();
    ptx::pdl_wait();
    __shared__ double red[256];
    double acc = 0.0;
    for (int i = threadIdx.x; i < nparts; i += blockDim.x) acc += a.partial[i];
    red[threadIdx.x] = acc;
    __syncthreads();
    for (int w = 128; w > 0; w >>= 1) {
        if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        const float mean = a.n > 0 ? static_cast<float>(red[0] / static_cast<double>(a.n)) : 0.0f;
        const float s = (mean > 0.0f && isfinite(mean)) ? __fdiv_rn(a.target, mean) : 0.0f;
        *a.s = s;
        if (a.s_out) *a.s_out = s;
    }
}

__global__ void __launch_bounds__(256) tern_sr4_update(const Sr4Args a) {
    ptx::pdl_trigger();
    ptx::pdl_wait();
    const float s = *a.s;
    const int64_t groups = a.n / 16;
    const int64_t nth = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (int64_t g = tid; g < groups; g += nth) {
        const int64_t e0 = g * 16;
        int4 qv = *reinterpret_cast<const int4*>(a.q + e0);
        const float4* gp = reinterpret_cast<const float4*>(a.gq + e0);
        float gv[16];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float4 f = __ldcs(gp + k);
            gv[4 * k] = f.x;
            gv[4 * k + 1] = f.y;
            gv[4 * k + 2] = f.z;
            gv[4 * k + 3] = f.w;
        }
        int8_t* qb = reinterpret_cast<int8_t*>(&qv);
        uint64_t z = sr4_counter(a, e0);
#pragma unroll
        for (int j = 0; j < 16; ++j, z += kG) qb[j] = sr4_one(a, qb[j], gv[j], s, z);
        *reinterpret_cast<int4*>(a.q + e0) = qv;
    }
    const int64_t t = groups * 16 + tid;   // scalar tail
    if (t < a.n) a.q[t] = sr4_one(a, a.q[t], a.gq[t], s, sr4_counter(a, t));
}

}  // namespace tern

using namespace tern;

extern "C" size_t tern_sr4_workspace(int64_t numel) {
    if (numel < 0) return 0;
    return kAbsumBlocks * sizeof(double) + 16;
}

extern "C" int tern_sr4_step(int8_t* q, const float* gq, int64_t numel, float inv_bs, float target_step,
                             uint64_t seed, int64_t idx_base, uint64_t counter, int q_clamp, int use_dither,
                             float* s_out, void* workspace, size_t ws_bytes, void* stream) {
    if (numel < 0 || q_clamp < 1 || q_clamp > 127 || idx_base < 0) return TERN_ERR_ARG;
    if (numel == 0) return TERN_OK;
    if (!q || !gq || !workspace) return TERN_ERR_ARG;
    if (!aligned16(q) || !aligned16(gq) || !aligned16(workspace)) return TERN_ERR_ALIGN;
    if (ws_bytes < tern_sr4_workspace(numel)) return TERN_ERR_WORKSPACE;
    int num_sms = 0;
    if (int st = check_device(&num_sms)) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    Sr4Args a;
    a.q = q;
    a.gq = gq;
    a.n = numel;
    a.inv_bs = inv_bs;
    a.target = target_step;
    a.key = mix64(seed ^ (counter * kG));
    a.idx_base = idx_base;
    a.clamp = q_clamp;
    a.dither = use_dither ? 1 : 0;
    a.partial = static_cast<double*>(workspace);
    a.s = reinterpret_cast<float*>(static_cast<char*>(workspace) + kAbsumBlocks * sizeof(double));
    a.s_out = s_out;
    const int nparts = static_cast<int>(numel < kAbsumBlocks ? numel : kAbsumBlocks);
    if (int st = launch_pdl(tern_sr4_absum, dim3(nparts), dim3(256), 0, s, a)) return st;
    if (int st = launch_pdl(tern_sr4_finalize, dim3(1), dim3(256), 0, s, a, nparts)) return st;
    const int64_t want = (numel / 16 + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    const unsigned grid = static_cast<unsigned>(want < 1 ? 1 : (want < cap ? want : cap));
    return launch_pdl(tern_sr4_update, dim3(grid), dim3(256), 0, s, a);
}

// ===================================================================== SR4 health panel
//
// Counts over the post-step accumulator of one weight (page "train_gpu.cu",
// sr4_panel_compute): ternary -1 / 0 / +1, rail (|q| == clamp), dead (|q| <
// theta) and churn (ternary differs from the previous 2-bit tiles), plus the
// scale's min / mean / max.  The page copies q and scale to the host and loops
// there; here one streaming pass over q (and the previous packed tiles) counts
// with byte-SIMD compares (four 16-byte loads in flight per thread), warp sums
// and one integer atomic per warp and counter (integer sums, so the result does
// not depend on the order), and one CTA reduces the scale in a fixed order.

namespace tern {
namespace {

struct PanelArgs {
    const int8_t* q;
    const uint32_t* prev;        // [K*N/16] previous packed tiles, or null
    const float* scale;
    int64_t groups;
    int64_t N;
    uint32_t th_pos, th_neg, cl;   // theta, -theta, clamp in every byte
    unsigned long long* counts;  // [6]
    double* sstats;              // [3]
};

}  // namespace

namespace {

// Counts of one 16-weight group (one 16-byte load) into c[0..5].
__device__ __forceinline__ void panel_group(const PanelArgs& a, const int4 raw, const uint32_t prev, uint32_t (&c)[6]) {
    const uint32_t w[4] = {static_cast<uint32_t>(raw.x), static_cast<uint32_t>(raw.y), static_cast<uint32_t>(raw.z),
                           static_cast<uint32_t>(raw.w)};
    uint32_t code = 0;
    uint32_t npos = 0, nneg = 0, nrail = 0, ndead = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t pos = __vcmpges4(w[k], a.th_pos);
        const uint32_t neg = __vcmples4(w[k], a.th_neg);
        const uint32_t mag = __vabs4(w[k]);             // |q| per byte (-128 stays 0x80, i.e. 128)
        npos += __popc(pos & 0x01010101u);
        nneg += __popc(neg & 0x01010101u);
        nrail += __popc(__vcmpeq4(mag, a.cl) & 0x01010101u);
        ndead += __popc(__vcmpltu4(mag, a.th_pos) & 0x01010101u);
        uint32_t x = (pos & 0x01010101u) | (neg & 0x03030303u);
        x = (x | (x >> 6) | (x >> 12) | (x >> 18)) & 0xFFu;
        code |= x << (8 * k);
    }
    c[0] += nneg;
    c[1] += 16 - npos - nneg;
    c[2] += npos;
    c[3] += nrail;
    c[4] += ndead;
    if (a.prev) {
        const uint32_t d = code ^ prev;
        c[5] += __popc((d | (d >> 1)) & 0x55555555u);    // 2-bit fields that differ
    }
}

}  // namespace

// Four groups per thread per pass, their loads issued before any is used; 32-bit
// counts per thread (at most 16 per group), 64-bit once per warp.
__global__ void __launch_bounds__(256) tern_panel_counts(const PanelArgs a) {
    ptx::pdl_trigger();
    ptx::pdl_wait();
    constexpr int U = 4;
    uint32_t c[6] = {0, 0, 0, 0, 0, 0};
    const int64_t nth = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int4* q4 = reinterpret_cast<const int4*>(a.q);
    for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; base < a.groups;
         base += nth * U) {
        int4 raw[U];
        uint32_t prev[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t gi = base + u * nth;
            raw[u] = make_int4(0, 0, 0, 0);
            prev[u] = 0;
            if (gi < a.groups) {
                raw[u] = __ldcs(q4 + gi);
                if (a.prev) prev[u] = __ldcs(a.prev + gi);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (base + u * nth < a.groups) panel_group(a, raw[u], prev[u], c);
    }
#pragma unroll
    for (int k = 0; k < 6; ++k) {
        unsigned long long v = c[k];
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if ((threadIdx.x & 31) == 0 && v) atomicAdd(a.counts + k, v);
    }
}

__global__ void __launch_bounds__(256) tern_panel_scale(const PanelArgs a) {
    ptx::pdl_trigger();
    ptx::pdl_wait();
    __shared__ double smin[256], smax[256], ssum[256];
    double mn = 0.0, mx = 0.0, sm = 0.0;
    bool any = false;
    for (int64_t c = threadIdx.x; c < a.N; c += blockDim.x) {
        const double s = a.scale[c];
        mn = any ? fmin(mn, s) : s;
        mx = any ? fmax(mx, s) : s;
        sm += s;
        any = true;
    }
    smin[threadIdx.x] = any ? mn : INFINITY;
    smax[threadIdx.x] = any ? mx : -INFINITY;
    ssum[threadIdx.x] = sm;
    __syncthreads();
    for (int w = 128; w > 0; w >>= 1) {
        if (threadIdx.x < w) {
            smin[threadIdx.x] = fmin(smin[threadIdx.x], smin[threadIdx.x + w]);
            smax[threadIdx.x] = fmax(smax[threadIdx.x], smax[threadIdx.x + w]);
            ssum[threadIdx.x] += ssum[threadIdx.x + w];
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        a.sstats[0] = smin[0];
        a.sstats[1] = ssum[0] / static_cast<double>(a.N);
        a.sstats[2] = smax[0];
    }
}

}  // namespace tern

extern "C" int tern_sr4_panel(const int8_t* q, const uint32_t* packed_prev, const float* scale, int64_t K,
                              int64_t N, int theta, int q_clamp, unsigned long long* counts, double* scale_stats,
                              void* stream) {
    if (!q || !scale || !counts || !scale_stats) return TERN_ERR_ARG;
    if (K < 1 || N < 16 || K * N >= (1ll << 40) || theta < 1 || q_clamp < theta || q_clamp > 127)
        return TERN_ERR_ARG;
    if (N % 16) return TERN_ERR_ALIGN;
    if (!aligned16(q) || (packed_prev && !aligned16(packed_prev)) || !aligned16(counts)) return TERN_ERR_ALIGN;
    int num_sms = 0;
    if (int st = check_device(&num_sms)) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    PanelArgs a;
    a.q = q;
    a.prev = packed_prev;
    a.scale = scale;
    a.groups = K * N / 16;
    a.N = N;
    a.th_pos = static_cast<uint32_t>(static_cast<uint8_t>(theta)) * 0x01010101u;
    a.th_neg = static_cast<uint32_t>(static_cast<uint8_t>(-theta)) * 0x01010101u;
    a.cl = static_cast<uint32_t>(static_cast<uint8_t>(q_clamp)) * 0x01010101u;
    a.counts = counts;
    a.sstats = scale_stats;
    TERN_CUDA_TRY(cudaMemsetAsync(counts, 0, 6 * sizeof(unsigned long long), s));
    const int64_t want = (a.groups + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (int st = launch_pdl(tern_panel_counts, dim3(static_cast<unsigned>(want < cap ? want : cap)), dim3(256), 0, s, a))
        return st;
    return launch_pdl(tern_panel_scale, dim3(1), dim3(256), 0, s, a);
}
