// AdamW step on continuous fp32 parameters (page "train_gpu.cu": adamw_dev with
// bias corrections bc_i = 1 - beta_i^t and the is_adamw switch, used for every
// continuous parameter and, after the scale_lr/lr factor, for the per-column
// scales; page "heal_gpu.rs": eps added outside the square root).
//
// HBM-bound: 28 bytes per element (read w, g, m, v; write w, m, v).  Each
// thread handles 4 consecutive elements per iteration with 16-byte loads and
// stores; a grid of 8 CTAs per SM strides over the array, and a scalar tail
// covers n % 4.
#include <math.h>

#include "common.cuh"

namespace tern {

namespace {

struct AdamArgs {
    float* w;
    const float* g;
    float* m;
    float* v;
    int64_t n;
    float lr, b1, b2, omb1, omb2, eps, wd, gmul, bc1, bc2;
    int decoupled;
};

__device__ __forceinline__ void adam_one(const AdamArgs& a, float& w, float g, float& m, float& v) {
    float gi = g * a.gmul;
    if (!a.decoupled) gi = fmaf(a.wd, w, gi);
    m = a.b1 * m + a.omb1 * gi;
    v = a.b2 * v + a.omb2 * gi * gi;
    const float mhat = m / a.bc1;
    const float vhat = v / a.bc2;
    const float step = a.lr * mhat / (sqrtf(vhat) + a.eps);
    const float decay = a.decoupled ? a.lr * a.wd * w : 0.0f;
    w = w - decay - step;
}

}  // namespace

__global__ void __launch_bounds__(256) tern_adamw_kernel(const AdamArgs a) {
    ptx::pdl_trigger();
    ptx::pdl_wait();
    const int64_t n4 = a.n >> 2;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    float4* w4 = reinterpret_cast<float4*>(a.w);
    const float4* g4 = reinterpret_cast<const float4*>(a.g);
    float4* m4 = reinterpret_cast<float4*>(a.m);
    float4* v4 = reinterpret_cast<float4*>(a.v);
    for (int64_t i = tid; i < n4; i += stride) {
        float4 w = __ldcs(w4 + i);
        const float4 g = __ldcs(g4 + i);
        float4 m = __ldcs(m4 + i);
        float4 v = __ldcs(v4 + i);
        adam_one(a, w.x, g.x, m.x, v.x);
        adam_one(a, w.y, g.y, m.y, v.y);
        adam_one(a, w.z, g.z, m.z, v.z);
        adam_one(a, w.w, g.w, m.w, v.w);
        __stcs(w4 + i, w);
        __stcs(m4 + i, m);
        __stcs(v4 + i, v);
    }
    const int64_t t = (n4 << 2) + tid;
    if (t < a.n) {
        float w = a.w[t], m = a.m[t], v = a.v[t];
        adam_one(a, w, a.g[t], m, v);
        a.w[t] = w;
        a.m[t] = m;
        a.v[t] = v;
    }
}

}  // namespace tern

using namespace tern;

extern "C" int adamw_step(float* w, const float* g, float* m, float* v, int64_t n, int t, float lr, float b1,
                          float b2, float eps, float wd, float gmul, int decoupled, void* stream) {
    if (n < 0 || t < 1) return TERN_ERR_ARG;
    if (n == 0) return TERN_OK;
    if (!w || !g || !m || !v) return TERN_ERR_ARG;
    if (!aligned16(w) || !aligned16(g) || !aligned16(m) || !aligned16(v)) return TERN_ERR_ALIGN;
    int num_sms = 0;
    if (int st = check_device(&num_sms)) return st;
    AdamArgs a;
    a.w = w;
    a.g = g;
    a.m = m;
    a.v = v;
    a.n = n;
    a.lr = lr;
    a.b1 = b1;
    a.b2 = b2;
    a.omb1 = static_cast<float>(1.0 - static_cast<double>(b1));
    a.omb2 = static_cast<float>(1.0 - static_cast<double>(b2));
    a.eps = eps;
    a.wd = wd;
    a.gmul = gmul;
    a.bc1 = static_cast<float>(1.0 - pow(static_cast<double>(b1), static_cast<double>(t)));
    a.bc2 = static_cast<float>(1.0 - pow(static_cast<double>(b2), static_cast<double>(t)));
    a.decoupled = decoupled ? 1 : 0;
    const int64_t want = ((n >> 2) + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    const unsigned grid = static_cast<unsigned>(want < 1 ? 1 : (want < cap ? want : cap));
    return launch_pdl(tern_adamw_kernel, dim3(grid), dim3(256), 0, static_cast<cudaStream_t>(stream), a);
}

// ===================================================================== several tensors per launch
//
// AdamW over up to TERN_ADAM_MAX_TENSORS tensors in one launch, with the
// per-step scalars {lr, bc1, bc2, gmul} read from device memory (page
// "train_gpu.cu", opt#3: the captured step reads them from the device buffer
// d_opt, so a replayed CUDA graph sees fresh values), and optionally the global
// gradient norm: a non-finite norm skips the whole step, a norm above max_norm
// scales every gradient by max_norm / norm (page "heal_gpu.rs": the skip and
// gmul = clip / gn; page "nvg_train.rs": grad_norm over every parameter).
//
// The tensors are cut into chunks of kChunk elements; the chunk table (prefix
// counts) travels in the kernel parameters, and each CTA finds a chunk's tensor
// by binary search.

namespace tern {
namespace {

constexpr int kChunk = 2048;        // AdamW chunk (elements)
constexpr int kSumChunk = 16384;    // sum-of-squares chunk (elements)

struct MultiArgs {
    int ntensors;
    int64_t nchunks;
    float b1, b2, omb1, omb2, eps, wd;
    int decoupled;
    const tern_adam_scalars* hp;
    const double* sumsq;
    float max_norm;
    int* skipped;
    int64_t first_chunk[TERN_ADAM_MAX_TENSORS + 1];
    int64_t n[TERN_ADAM_MAX_TENSORS];
    float* w[TERN_ADAM_MAX_TENSORS];
    const float* g[TERN_ADAM_MAX_TENSORS];
    float* m[TERN_ADAM_MAX_TENSORS];
    float* v[TERN_ADAM_MAX_TENSORS];
};

struct SumArgs {
    int ntensors;
    int64_t nchunks;
    double* partial;
    double* out;
    int64_t first_chunk[TERN_ADAM_MAX_TENSORS + 1];
    int64_t n[TERN_ADAM_MAX_TENSORS];
    const float* g[TERN_ADAM_MAX_TENSORS];
};

// Every launch's parameter block stays within 4 KB (the tables above are sized by
// TERN_ADAM_MAX_TENSORS), so all launches take the same driver path; a launch with
// a larger block (6 KB at 128 tensors), issued with programmatic dependent launch,
// was the one launch of that kind in a chain that stopped making progress.
static_assert(sizeof(MultiArgs) <= 4096 && sizeof(SumArgs) <= 4096, "kernel parameter block over 4 KB");

template <class A>
__device__ __forceinline__ int chunk_tensor(const A& a, int64_t ch) {
    int lo = 0, hi = a.ntensors - 1;   // last t with first_chunk[t] <= ch
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.first_chunk[mid] <= ch) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ void adam_elem(const MultiArgs& a, float lr, float bc1, float bc2, float gmul, float& w,
                                          float g, float& m, float& v) {
    float gi = __fmul_rn(g, gmul);
    if (!a.decoupled) gi = fmaf(a.wd, w, gi);
    m = a.b1 * m + a.omb1 * gi;
    v = a.b2 * v + a.omb2 * gi * gi;
    const float step = lr * (m / bc1) / (sqrtf(v / bc2) + a.eps);
    const float decay = a.decoupled ? lr * a.wd * w : 0.0f;
    w = w - decay - step;
}

}  // namespace

__global__ void __launch_bounds__(256) tern_adamw_multi_kernel(const __grid_constant__ MultiArgs a) {
    ptx::pdl_trigger();
    ptx::pdl_wait();
    const tern_adam_scalars hp = *a.hp;
    float gmul = hp.gmul;
    if (a.sumsq) {
        const double norm = sqrt(*a.sumsq);
        const bool skip = !isfinite(norm);
        if (blockIdx.x == 0 && threadIdx.x == 0 && a.skipped) *a.skipped = skip ? 1 : 0;
        if (skip) return;
        if (a.max_norm > 0.0f && norm > static_cast<double>(a.max_norm))
            gmul = __fmul_rn(gmul, static_cast<float>(static_cast<double>(a.max_norm) / norm));
    } else if (blockIdx.x == 0 && threadIdx.x == 0 && a.skipped) {
        *a.skipped = 0;
    }
    for (int64_t ch = blockIdx.x; ch < a.nchunks; ch += gridDim.x) {
        const int t = chunk_tensor(a, ch);
        const int64_t off = (ch - a.first_chunk[t]) * kChunk;
        const int64_t cnt = min(static_cast<int64_t>(kChunk), a.n[t] - off);
        float* w = a.w[t] + off;
        const float* g = a.g[t] + off;
        float* m = a.m[t] + off;
        float* v = a.v[t] + off;
        const int n4 = static_cast<int>(cnt >> 2);
        for (int i = threadIdx.x; i < n4; i += blockDim.x) {
            float4 w4 = __ldcs(reinterpret_cast<float4*>(w) + i);
            const float4 g4 = __ldcs(reinterpret_cast<const float4*>(g) + i);
            float4 m4 = __ldcs(reinterpret_cast<float4*>(m) + i);
            float4 v4 = __ldcs(reinterpret_cast<float4*>(v) + i);
            adam_elem(a, hp.lr, hp.bc1, hp.bc2, gmul, w4.x, g4.x, m4.x, v4.x);
            adam_elem(a, hp.lr, hp.bc1, hp.bc2, gmul, w4.y, g4.y, m4.y, v4.y);
            adam_elem(a, hp.lr, hp.bc1, hp.bc2, gmul, w4.z, g4.z, m4.z, v4.z);
            adam_elem(a, hp.lr, hp.bc1, hp.bc2, gmul, w4.w, g4.w, m4.w, v4.w);
            __stcs(reinterpret_cast<float4*>(w) + i, w4);
            __stcs(reinterpret_cast<float4*>(m) + i, m4);
            __stcs(reinterpret_cast<float4*>(v) + i, v4);
        }
        const int j = n4 * 4 + threadIdx.x;
        if (j < cnt) {
            float wj = w[j], mj = m[j], vj = v[j];
            adam_elem(a, hp.lr, hp.bc1, hp.bc2, gmul, wj, g[j], mj, vj);
            w[j] = wj;
            m[j] = mj;
            v[j] = vj;
        }
    }
}

// Per-chunk fp64 sums of squares (fixed chunking and order), then one CTA sums
// the chunk partials in a fixed order.
__global__ void __launch_bounds__(256) tern_sumsq_chunks(const __grid_constant__ SumArgs a) {
    ptx::pdl_trigger();
    ptx::pdl_wait();
    __shared__ double red[256];
    for (int64_t ch = blockIdx.x; ch < a.nchunks; ch += gridDim.x) {
        const int t = chunk_tensor(a, ch);
        const int64_t off = (ch - a.first_chunk[t]) * kSumChunk;
        const int64_t cnt = min(static_cast<int64_t>(kSumChunk), a.n[t] - off);
        const float* g = a.g[t] + off;
        double acc = 0.0;
        for (int64_t i = threadIdx.x; i < cnt; i += blockDim.x) {
            const double x = g[i];
            acc += x * x;
        }
        red[threadIdx.x] = acc;
        __syncthreads();
        for (int s = 128; s > 0; s >>= 1) {
            if (threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
            __syncthreads();
        }
        if (threadIdx.x == 0) a.partial[ch] = red[0];
        __syncthreads();
    }
}

__global__ void __launch_bounds__(256) tern_sumsq_final(const double* __restrict__ partial, int64_t nparts,
                                                        double* __restrict__ out) {
    ptx::pdl_trigger();
    ptx::pdl_wait();
    __shared__ double red[256];
    double acc = 0.0;
    for (int64_t i = threadIdx.x; i < nparts; i += blockDim.x) acc += partial[i];
    red[threadIdx.x] = acc;
    __syncthreads();
    for (int s = 128; s > 0; s >>= 1) {
        if (threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
        __syncthreads();
    }
    if (threadIdx.x == 0) *out = red[0];
}

namespace {
int64_t count_chunks(const int64_t* n, int ntensors, int64_t chunk, int64_t* first) {
    int64_t total = 0;
    for (int t = 0; t < ntensors; ++t) {
        if (first) first[t] = total;
        total += (n[t] + chunk - 1) / chunk;
    }
    if (first) first[ntensors] = total;
    return total;
}
}  // namespace

}  // namespace tern

extern "C" size_t tern_grad_sumsq_workspace(const int64_t* n, int ntensors) {
    if (!n || ntensors < 1 || ntensors > TERN_ADAM_MAX_TENSORS) return 0;
    for (int t = 0; t < ntensors; ++t)
        if (n[t] < 0) return 0;
    return static_cast<size_t>(count_chunks(n, ntensors, kSumChunk, nullptr) + 1) * sizeof(double);
}

extern "C" int tern_grad_sumsq(const float* const* g, const int64_t* n, int ntensors, double* sumsq,
                               void* workspace, size_t ws_bytes, void* stream) {
    if (!g || !n || !sumsq || ntensors < 1 || ntensors > TERN_ADAM_MAX_TENSORS) return TERN_ERR_ARG;
    SumArgs a{};
    a.ntensors = ntensors;
    for (int t = 0; t < ntensors; ++t) {
        if (n[t] < 0 || (n[t] > 0 && !g[t])) return TERN_ERR_ARG;
        a.n[t] = n[t];
        a.g[t] = g[t];
    }
    a.nchunks = count_chunks(n, ntensors, kSumChunk, a.first_chunk);
    if (!workspace || !aligned16(workspace)) return workspace ? TERN_ERR_ALIGN : TERN_ERR_ARG;
    if (ws_bytes < tern_grad_sumsq_workspace(n, ntensors)) return TERN_ERR_WORKSPACE;
    int num_sms = 0;
    if (int st = check_device(&num_sms)) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    a.partial = static_cast<double*>(workspace);
    a.out = sumsq;
    if (a.nchunks > 0) {
        const int64_t grid = a.nchunks < 8 * num_sms ? a.nchunks : 8 * num_sms;
        if (int st = launch_pdl(tern_sumsq_chunks, dim3(static_cast<unsigned>(grid)), dim3(256), 0, s, a)) return st;
    }
    return launch_pdl(tern_sumsq_final, dim3(1), dim3(256), 0, s, static_cast<const double*>(a.partial), a.nchunks, sumsq);
}

extern "C" int adamw_step_multi(float* const* w, const float* const* g, float* const* m, float* const* v,
                                const int64_t* n, int ntensors, const tern_adam_scalars* scalars, float b1, float b2,
                                float eps, float wd, int decoupled, const double* sumsq, float max_norm,
                                int* skipped, void* stream) {
    if (!w || !g || !m || !v || !n || !scalars || ntensors < 1 || ntensors > TERN_ADAM_MAX_TENSORS)
        return TERN_ERR_ARG;
    MultiArgs a{};
    a.ntensors = ntensors;
    for (int t = 0; t < ntensors; ++t) {
        if (n[t] < 0) return TERN_ERR_ARG;
        if (n[t] > 0 && (!w[t] || !g[t] || !m[t] || !v[t])) return TERN_ERR_ARG;
        if (!aligned16(w[t]) || !aligned16(g[t]) || !aligned16(m[t]) || !aligned16(v[t])) return TERN_ERR_ALIGN;
        a.n[t] = n[t];
        a.w[t] = w[t];
        a.g[t] = g[t];
        a.m[t] = m[t];
        a.v[t] = v[t];
    }
    a.nchunks = count_chunks(n, ntensors, kChunk, a.first_chunk);
    int num_sms = 0;
    if (int st = check_device(&num_sms)) return st;
    a.b1 = b1;
    a.b2 = b2;
    a.omb1 = static_cast<float>(1.0 - static_cast<double>(b1));
    a.omb2 = static_cast<float>(1.0 - static_cast<double>(b2));
    a.eps = eps;
    a.wd = wd;
    a.decoupled = decoupled ? 1 : 0;
    a.hp = scalars;
    a.sumsq = sumsq;
    a.max_norm = max_norm;
    a.skipped = skipped;
    const int64_t grid = a.nchunks < 1 ? 1 : (a.nchunks < 8 * num_sms ? a.nchunks : 8 * num_sms);
    return launch_pdl(tern_adamw_multi_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0,
                      static_cast<cudaStream_t>(stream), a);
}
