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
    tern_adamw_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(a);
    TERN_CUDA_TRY(cudaGetLastError());
    return TERN_OK;
}
