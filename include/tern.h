/*
 * tern.h — C ABI of the GB300 (sm_103a) ternary-weight linear layer library.
 *
 * The layer (page "train_gpu.cu", header comment "Optimizer split" and the device
 * glue kernels tg_tern_from_q / tg_apply_scale / tg_gq / tg_scale_grad):
 *
 *   ternary(q)[r,c] = +1 if q >= theta, -1 if q <= -theta, else 0
 *   W_eff[r,c]      = scale[c] * ternary(q)[r,c]        (row-major [K][N])
 *   Y               = X * W_eff                          (forward)
 *   dX              = dY * W_eff^T                       (input gradient)
 *   gq[r,c]         = (X^T * dY)[r,c] * scale[c]         (straight-through gradient)
 *   sgrad[c]        = sum_r (X^T * dY)[r,c] * ternary(q)[r,c]   (scale gradient)
 *
 * followed by AdamW on continuous parameters, the scales included (same page,
 * resident optimizer launchers: adamw_dev and its bias corrections 1 - beta^t).
 *
 * Shapes: M tokens, K input features (rows r of q), N output features (columns
 * c of q).  Every matrix is row-major and dense.  Element types: X, dY bf16 (as
 * uint16 bit patterns), q int8, scale and every output fp32.
 *
 * Ownership and ordering: the caller allocates and owns every buffer (device
 * memory unless stated otherwise).  No call allocates, frees or synchronises.
 * Each call enqueues its kernels on `stream` (a cudaStream_t; NULL is the
 * legacy default stream) and returns once they are enqueued; outputs are valid
 * when the stream reaches that point.  Calls may be captured into a CUDA graph
 * after the first call on a device (which loads the driver's tensor-map
 * encoder).  Inputs must not alias outputs.
 *
 * Errors: every call returns TERN_OK (0) or a negative status, checks its
 * arguments before enqueueing anything, and never exits the process.  Inside
 * the GEMM kernels, every wait on the tensor-core pipeline (an mbarrier between
 * the TMA producer, the MMA issuer and the epilogue) gives up after a bounded
 * time and records TERN_ERR_TIMEOUT in a device status word that
 * tern_device_status() reads back.  Three waits of a GEMM's set-up have no
 * bound, because the hardware gives none: the tensor-memory allocation
 * (tcgen05.alloc), the cluster barrier of a CTA pair and the dependent-launch
 * wait.  The GEMMs are launched with full stream serialization (no
 * programmatic dependent launch), so a GEMM starts only after every earlier
 * kernel on its stream has completed and those waits never wait on another grid.
 */
#ifndef TERN_H
#define TERN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TERN_OK 0
#define TERN_ERR_ARG (-1)         /* null pointer, non-positive size, theta < 1, clamp < theta */
#define TERN_ERR_ALIGN (-2)       /* K or N not a multiple of 16, pointer not 16-byte aligned */
#define TERN_ERR_CUDA (-3)        /* a CUDA runtime/driver call failed (launch, attribute, map) */
#define TERN_ERR_TIMEOUT (-4)     /* a bounded device-side wait gave up */
#define TERN_ERR_WORKSPACE (-5)   /* workspace smaller than tern_linear_bwd_workspace() */
#define TERN_ERR_DEVICE (-6)      /* current device is not an sm_103 (GB300) part */
#define TERN_ERR_SCRATCH_LIMIT (-7) /* problem larger than tern_linear_bwd_noalloc's built-in scratch */

/* Weight operands produced by tern_materialize from q and scale; caller-owned
 * device buffers.  Any pointer may be NULL to skip that output; the GEMM calls
 * state which ones they read. */
typedef struct tern_tiles {
    uint32_t* packed;   /* [K][N/16] 2-bit codes, element (r,c) at word r*(N/16)+c/16,
                           bits 2*(c%16): 0 -> 00, +1 -> 01, -1 -> 11 (10 never written) */
    uint16_t* t_bf16;   /* [K][N] bf16 of ternary(q): 0x0000, 0x3F80, 0xBF80 (forward operand) */
    uint16_t* whi_bf16; /* [K][N] bf16 of s_hi[c]*ternary(q), s_hi = bf16_rne(scale[c]) */
    uint16_t* wlo_bf16; /* [K][N] bf16 of s_lo[c]*ternary(q), s_lo = bf16_rne(scale[c]-s_hi) */
    /* The fp16 + e4m3 split of the dX operand (read by tern_linear_bwd_ex with
     * TERN_BWD_DX_SPLIT8).  scale[c] = a_c * 2^e_c, e_c = floor(log2|scale[c]|), a_c in
     * +-[1,2) (a_c = 0 for a zero scale); h_c = binary16_rne(a_c), l_c =
     * e4m3_rne_satfinite(2^7 * (a_c - h_c)) (OCP E4M3: bias 7, largest 448), so that
     * h_c + 2^-7 l_c = a_c within 2^-15 |a_c|.  A zero weight is +0 in both planes; a
     * negative one flips the sign bit. */
    uint16_t* whi_f16;  /* [K][N] binary16 of h_c*ternary(q) */
    uint8_t* wlo_e4m3;  /* [K][N] e4m3 of l_c*ternary(q) */
} tern_tiles;

#define TERN_TILE_PACKED 0
#define TERN_TILE_T 1
#define TERN_TILE_WHI 2
#define TERN_TILE_WLO 3
#define TERN_TILE_WHI16 4
#define TERN_TILE_WLO8 5

/* Bytes of one tern_tiles buffer (`which` = TERN_TILE_*) for a K x N weight; 0 on bad args. */
size_t tern_tiles_bytes(int64_t K, int64_t N, int which);

/*
 * Ternarise and encode one weight matrix (page "train_gpu.cu", tg_tern_from_q,
 * and the accumulator clamp SR4_Q_CLAMP).
 *   q         [K][N] int8 accumulator (device, read)
 *   q_clamped [K][N] int8, min(max(q,-q_clamp),q_clamp) (device, written; NULL to skip;
 *             may equal q for an in-place clamp)
 *   scale     [N] fp32 (device, read; may be NULL when out has no hi/lo or fp16/e4m3 planes)
 *   out       tiles to write (host struct of device pointers; NULL members skipped)
 *   theta >= 1, q_clamp >= theta (clamping then keeps every ternary value).
 * K >= 1, N >= 16 with N % 16 == 0; every pointer 16-byte aligned.  Bit-exact.
 */
int tern_materialize(const int8_t* q, int8_t* q_clamped, const float* scale, int64_t K, int64_t N,
                     int theta, int q_clamp, const tern_tiles* out, void* stream);

/*
 * tern_materialize for several weights in one call: one launch per set of requested
 * encodings (16 weights at a time), each weight on its own range of blocks, so that
 * the small weights of one block do not each pay a launch.  Same results, rules and
 * errors as the single-weight call, weight by weight; nothing is enqueued if any
 * weight's arguments are bad.  theta and q_clamp are shared by every weight.  The
 * pages materialise each weight in its own passes; the grouping is this library's.
 */
typedef struct tern_mat_layer {
    const int8_t* q;         /* [K][N] int8 accumulator (device, read) */
    int8_t* q_clamped;       /* [K][N] clamped q (device, written; NULL to skip; may equal q) */
    const float* scale;      /* [N] fp32 (device; may be NULL without hi/lo planes) */
    const tern_tiles* out;   /* tiles to write (host struct of device pointers) */
    int64_t K, N;
} tern_mat_layer;
int tern_materialize_grouped(const tern_mat_layer* layers, int count, int theta, int q_clamp, void* stream);

/*
 * Forward: Y[m][c] = scale[c] * sum_r X[m][r] * T[r][c] (page "train_gpu.cu",
 * header comment: W_eff = scale[c]*ternary(q); the forward GEMM itself is the
 * off-page fm_forward).  The scale is applied in the epilogue, so W_eff is never
 * formed.  Reads W->t_bf16; with W->t_bf16 NULL it reads W->packed instead and
 * expands the 2-bit codes into bf16 operand tiles inside the GEMM (same result,
 * bit for bit; N must then be a multiple of 64, else TERN_ERR_ALIGN).  With neither
 * plane given: TERN_ERR_ARG.
 *   X [M][K] bf16 (device), scale [N] fp32 (device), Y [M][N] fp32 (device, written).
 * M >= 1; K, N >= 16 and multiples of 16; pointers 16-byte aligned.
 * Tensor cores, bf16 x {-1,0,+1} products (exact), fp32 accumulation.
 */
int tern_linear_fwd(const uint16_t* X, const tern_tiles* W, const float* scale, float* Y, int64_t M,
                    int64_t K, int64_t N, void* stream);

/*
 * Device workspace of tern_linear_bwd, in bytes.
 *   tern_linear_bwd_workspace_min: the sgrad partials, the least a call computing
 *     sgrad accepts (ceil(K/128)*4*N floats).
 *   tern_linear_bwd_workspace: the partials plus room for the split tail of the G
 *     GEMM (at most 128 partial tiles of 256 x 256 fp32): when the last wave of G
 *     tiles would leave SMs idle, or a small K x N has too few tiles, the
 *     remaining tiles are split along the token axis and reduced in a fixed
 *     order.  A workspace between the two sizes runs without the split.
 */
size_t tern_linear_bwd_workspace_min(int64_t M, int64_t K, int64_t N);
size_t tern_linear_bwd_workspace(int64_t M, int64_t K, int64_t N);

/*
 * Backward (page "train_gpu.cu": the backward GEMMs are the off-page fm_backward;
 * tg_gq and tg_scale_grad give gq and sgrad from grad = X^T * dY).
 *   dX[m][r]  = sum_c dY[m][c] * scale[c] * T[r][c]   fp32 [M][K]  (NULL to skip)
 *               computed as dY*W_hi^T + dY*W_lo^T (reads W->whi_bf16, W->wlo_bf16; with both
 *               NULL it reads W->packed and expands W_hi / W_lo from the codes and a
 *               per-column s_hi / s_lo table inside the GEMM: the same bits, so the same dX,
 *               at the cost of converter work in the GEMM; then N % 64 == 0 (else
 *               TERN_ERR_ALIGN) and a workspace of at least 4*N bytes are needed)
 *   gq[r][c]  = G[r][c] * scale[c], G = X^T * dY      fp32 [K][N]  (NULL to skip)
 *   sgrad[c]  = sum_r G[r][c] * T[r][c]               fp32 [N]    (NULL to skip;
 *               reads W->packed)
 * gq and sgrad come from one fused epilogue of the G GEMM; G itself is never
 * stored.  sgrad is reduced over r in a fixed order (deterministic run to run).
 * At least one of dX, gq, sgrad must be given; with gq and sgrad both NULL the
 * G GEMM is not run, with dX NULL the dX GEMM is not run.
 *   X [M][K] bf16, dY [M][N] bf16, scale [N] fp32: device, read.
 *   workspace: device, 16-byte aligned, contents ignored and overwritten; at least
 *   tern_linear_bwd_workspace_min(M,K,N) bytes when sgrad is requested (else may
 *   be NULL); tern_linear_bwd_workspace(M,K,N) bytes enable the split G tail.
 * Same shape rules as the forward.
 */
int tern_linear_bwd(const uint16_t* X, const uint16_t* dY, const tern_tiles* W, const float* scale,
                    float* dX, float* gq, float* sgrad, void* workspace, size_t ws_bytes, int64_t M,
                    int64_t K, int64_t N, void* stream);

/*
 * tern_linear_bwd with flags.  TERN_BWD_ACCUMULATE adds this call's gq and sgrad
 * to the values already stored (dX is still overwritten): the gradient of B
 * micro-batches is the sum of B calls, the first without the flag (page
 * "train_gpu.cu": the B > 1 path accumulates every gradient over micro-batches
 * before the optimizer step and scales by 1/B; here the 1/B goes into
 * tern_sr4_step's inv_bs and AdamW's gmul).  Unknown flag bits: TERN_ERR_ARG.
 *
 * TERN_BWD_DX_SPLIT8 computes dX from the fp16 + e4m3 split instead of the bf16
 * hi/lo split: it reads W->whi_f16 and W->wlo_e4m3 (not whi_bf16 / wlo_bf16) and
 * first splits dY, per row m, into binary16 dY[m][c]*2^(e_c-e_m) and e4m3
 * dY[m][c]*2^(e_c-e_m-7) copies, e_m chosen so that the row's largest
 * |dY[m][c]|*2^e_c lands in [2^14, 2^15); the GEMM is then one binary16 pass and one
 * e4m3 pass (twice the bf16 rate) into one accumulator, times 2^e_m.  The workspace
 * must hold the split: at least tern_linear_bwd_workspace_ex(M, K, N, flags) bytes
 * (the copies are consumed before the G GEMM, which reuses the same bytes).
 * Error of each dX[m][r] against the exact sum, besides fp32 accumulation:
 *   <= 6.3e-5 * sum_c |dY[m][c] scale[c] T[r][c]|
 *      + 4.3e-9 * max_c |dY[m][c] scale[c]| * #{c : T[r][c] != 0}
 * (the second term from dY values more than 2^13 below the row's largest, whose e4m3
 * copy loses bits).  The bf16 split's bound is 2^-16 of the first sum alone.
 */
#define TERN_BWD_ACCUMULATE 1u
#define TERN_BWD_DX_SPLIT8 2u
size_t tern_linear_bwd_workspace_ex(int64_t M, int64_t K, int64_t N, unsigned flags);
int tern_linear_bwd_ex(const uint16_t* X, const uint16_t* dY, const tern_tiles* W, const float* scale,
                       float* dX, float* gq, float* sgrad, void* workspace, size_t ws_bytes, int64_t M,
                       int64_t K, int64_t N, unsigned flags, void* stream);

/*
 * Grouped calls: several independent layers (for example the four token-mixing
 * projections of a block, which read the same input) in one call, so that the
 * tiles of small layers fill the GPU together.  The paper runs each projection
 * as its own GEMM (page "train_gpu.cu", the per-layer GEMM calls of the
 * forward and backward); the grouping is this library's.  One layer:
 */
typedef struct tern_layer {
    const uint16_t* X;    /* [M][K] bf16, device */
    const uint16_t* dY;   /* [M][N] bf16, device (backward only) */
    const tern_tiles* W;  /* the layer's tiles: host struct of device pointers */
    const float* scale;   /* [N] fp32, device */
    float* Y;             /* [M][N] fp32, device (forward only) */
    float* dX;            /* [M][K] fp32, device (backward; NULL skips it) */
    float* gq;            /* [K][N] fp32, device (backward; NULL skips it) */
    float* sgrad;         /* [N] fp32, device (backward; NULL skips it) */
    int64_t M, K, N;
    uint16_t* Y_bf16;     /* [M][N] bf16 (round to nearest even) copy of Y, device, or NULL */
    uint16_t* dX_bf16;    /* [M][K] bf16 copy of dX, device, or NULL */
} tern_layer;

/*
 * tern_linear_fwd for every layer of `layers` (host array of count >= 1 layers;
 * each layer's own shape).  Same rules, errors and results as the single-layer
 * call, layer by layer; nothing is enqueued if any layer's arguments are bad.
 * Y_bf16, when given, receives Y rounded to bf16 from the same epilogue, so the
 * next layer of a chain reads its input without a separate cast; Y may then be
 * NULL.
 * Layers are launched up to eight at a time; a layer's Y must not overlap
 * another layer's inputs.
 * Known issue of an earlier build: with the GEMMs launched by programmatic
 * dependent launch (their set-up overlapping the previous kernel), a process that
 * had first run long single-layer steps of a large projection and then a sequence
 * of eager grouped calls stalled, with one CTA pair of a GEMM unable to finish its
 * set-up (tensor-memory allocation, cluster barrier).  The cause was not found.
 * The GEMMs are now launched with full stream serialization, so that set-up no
 * longer overlaps any other grid; tern_device_diagnostics reports the state
 * should a stall happen.
 */
int tern_linear_fwd_grouped(const tern_layer* layers, int count, void* stream);

/*
 * tern_linear_bwd_ex for every layer.  One workspace (device, 16-byte aligned,
 * contents ignored) of at least the sum over layers of the sgrad partials
 * (each tern_linear_bwd_workspace_min rounded up to 256 bytes) serves all;
 * tern_linear_bwd_grouped_workspace() bytes (0 on bad shapes) add room for
 * splitting the G tiles of small layers along the token axis.  dX equals the
 * single-layer call's; gq and sgrad equal it up to the order of fp32 sums.
 * dX_bf16 (with or without dX) receives dX rounded to bf16: the dY of the layer
 * before in a chain.
 * A layer that asks for dX needs the hi/lo planes here (the expansion from the codes
 * and the fp16 + e4m3 split are single-layer options of tern_linear_bwd_ex).
 * flags: 0 or TERN_BWD_ACCUMULATE (every layer).  Errors as tern_linear_bwd_ex;
 * a NULL workspace is TERN_ERR_WORKSPACE.
 */
size_t tern_linear_bwd_grouped_workspace(const tern_layer* layers, int count);
int tern_linear_bwd_grouped(const tern_layer* layers, int count, void* workspace, size_t ws_bytes,
                            unsigned flags, void* stream);

/*
 * tern_linear_bwd for callers that cannot allocate device memory.  The paper
 * has no counterpart of this call; it is a convenience of this library.
 *
 * Same arguments, outputs and rules as tern_linear_bwd, minus the workspace.
 * Some callers cannot call cudaMalloc (for example a plugin whose host program
 * owns every device allocation, or a loop that must not pay cudaMalloc's
 * device-wide synchronisation), so they cannot provide one.  This entry point
 * keeps the sgrad partials in a fixed array inside the library's device image
 * instead; it allocates nothing.
 *   Limit: tern_linear_bwd_workspace_min(M, K, N) <= TERN_NOALLOC_SCRATCH_BYTES
 *   (8 MiB: ceil(K/128)*4*N <= 2^21, e.g. K = 4096 with N <= 16384) when sgrad
 *   is requested, else TERN_ERR_SCRATCH_LIMIT and nothing is enqueued.
 *   Every GPU that loads the library holds the 8 MiB until the process exits.
 *   The first call on each device looks up the array's device address (with
 *   that device current); make it before any stream capture.
 *   All calls share the array: calls whose kernels overlap on a GPU race and
 *   corrupt each other's sgrad.  Order them on one stream (or with events).
 */
#define TERN_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
int tern_linear_bwd_noalloc(const uint16_t* X, const uint16_t* dY, const tern_tiles* W, const float* scale,
                            float* dX, float* gq, float* sgrad, int64_t M, int64_t K, int64_t N,
                            void* stream);

/*
 * AdamW on n fp32 elements (page "train_gpu.cu", adamw_dev: bias corrections
 * bc_i = 1 - beta_i^t, is_adamw; page "heal_gpu.rs": eps outside the root).
 *   g' = gmul*g (+ wd*w when decoupled == 0)
 *   m  = b1*m + (1-b1)*g';  v = b2*v + (1-b2)*g'^2
 *   w  = w - [decoupled] lr*wd*w - lr*(m/bc1)/(sqrt(v/bc2)+eps)      (decay uses the old w)
 * w, m, v updated in place; g read.  All device, 16-byte aligned; t >= 1; n >= 0
 * (n == 0 enqueues nothing).  gmul is the page's scale_lr/lr factor (1 for none).
 */
int adamw_step(float* w, const float* g, float* m, float* v, int64_t n, int t, float lr, float b1,
               float b2, float eps, float wd, float gmul, int decoupled, void* stream);

/*
 * Per-step AdamW scalars kept in device memory (page "train_gpu.cu", opt#3: the
 * captured training step reads {lr, bc1, bc2, scale_lr/lr} from a device buffer
 * so that a replayed CUDA graph sees fresh values).  bc_i = 1 - beta_i^t; gmul
 * multiplies the gradient.  The caller writes them before each step.
 */
typedef struct tern_adam_scalars {
    float lr, bc1, bc2, gmul;
} tern_adam_scalars;

/* Tensors per multi-tensor call; more tensors take several calls.  The bound keeps
 * each launch's parameter block (the per-tensor table) under 4 KB. */
#define TERN_ADAM_MAX_TENSORS 64

/*
 * Global gradient sum of squares over several tensors, fp64, in a fixed order
 * (page "train_gpu.cu": grad_l2_gpu; page "nvg_train.rs": grad_norm).
 *   g[t], n[t]: host arrays of ntensors (1..TERN_ADAM_MAX_TENSORS) device pointers
 *   and element counts; sumsq: device double, written.
 *   workspace: device, >= tern_grad_sumsq_workspace(n, ntensors) bytes, 16-byte aligned.
 */
size_t tern_grad_sumsq_workspace(const int64_t* n, int ntensors);
int tern_grad_sumsq(const float* const* g, const int64_t* n, int ntensors, double* sumsq, void* workspace,
                    size_t ws_bytes, void* stream);

/*
 * AdamW (same update as adamw_step) over ntensors tensors in one launch, reading
 * lr, bc1, bc2 and gmul from `scalars` in device memory.  When sumsq (device,
 * from tern_grad_sumsq) is given: a non-finite norm sqrt(sumsq) skips the whole
 * step (nothing is written); a norm above max_norm > 0 multiplies every gradient
 * by max_norm / norm (page "heal_gpu.rs": skip non-finite steps, gmul = clip / gn;
 * page "nvg_train.rs": adam's gmul).  skipped (device int, may be NULL) receives
 * 1 for a skipped step, else 0.
 *   w, g, m, v, n: host arrays of device pointers / element counts; every tensor
 *   16-byte aligned; 1 <= ntensors <= TERN_ADAM_MAX_TENSORS.
 */
int adamw_step_multi(float* const* w, const float* const* g, float* const* m, float* const* v, const int64_t* n,
                     int ntensors, const tern_adam_scalars* scalars, float b1, float b2, float eps, float wd,
                     int decoupled, const double* sumsq, float max_norm, int* skipped, void* stream);

/*
 * SR4 step on one weight's int4 accumulator (page "train_gpu.cu": sr4_dev calls
 * fc_sr4_scale<<<1,1>>>(gq, numel, inv_bs, target_step, d_s) then
 * fc_sr4_update(q, gq, numel, inv_bs, d_s, seed, idx_base, counter, q_clamp,
 * use_dither); the bodies are off the page, so this is the plainest reading of
 * those arguments):
 *   s   = target_step / mean_i |gq_i*inv_bs|                 (s = 0 when the mean is 0)
 *   q_i = clamp(q_i - floor((gq_i*inv_bs)*s + u_i), -q_clamp, q_clamp)
 * i.e. stochastic rounding of the descent step into the accumulator, with
 * u_i ~ U[0,1) from splitmix64 keyed by (seed, counter) at global index
 * idx_base + i (use_dither = 0: u_i = 1/2).  A non-finite step leaves q_i as is.
 *   q [numel] int8 (device, updated in place), gq [numel] fp32 (device, read).
 *   s_out: device float receiving s (NULL to skip).
 *   workspace: device, >= tern_sr4_workspace(numel) bytes, 16-byte aligned.
 * q and gq 16-byte aligned; numel >= 0; 1 <= q_clamp <= 127; idx_base >= 0.
 * The sum behind s is reduced in a fixed order (deterministic).
 */
size_t tern_sr4_workspace(int64_t numel);
int tern_sr4_step(int8_t* q, const float* gq, int64_t numel, float inv_bs, float target_step, uint64_t seed,
                  int64_t idx_base, uint64_t counter, int q_clamp, int use_dither, float* s_out,
                  void* workspace, size_t ws_bytes, void* stream);

/*
 * SR4 health panel of one weight (page "train_gpu.cu", sr4_panel_compute), from
 * the post-step q [K][N] and scale [N]:
 *   counts[0..5] = #ternary -1, #ternary 0, #ternary +1, #|q| == q_clamp (rail),
 *                  #|q| < theta (dead), #ternary differing from packed_prev (churn)
 *   scale_stats[0..2] = min, mean, max of scale (fp64)
 *   packed_prev: the previous 2-bit tiles [K][N/16] (from tern_materialize), or
 *   NULL (churn 0).  counts (device, 6 x u64, 16-byte aligned) is overwritten;
 *   scale_stats: device, 3 doubles.  Integer counts: the result is exact and
 *   does not depend on the launch.  Same shape rules as tern_materialize.
 */
int tern_sr4_panel(const int8_t* q, const uint32_t* packed_prev, const float* scale, int64_t K, int64_t N,
                   int theta, int q_clamp, unsigned long long* counts, double* scale_stats, void* stream);

/* Text of a status code (static storage). */
const char* tern_strerror(int status);

/*
 * Synchronise `stream`, then return TERN_ERR_TIMEOUT if any kernel since the last
 * clear gave up on a bounded wait, else TERN_OK (TERN_ERR_CUDA if the sync fails).
 * clear != 0 resets the device status word.  This is the one call that blocks.
 */
int tern_device_status(void* stream, int clear);

/*
 * Failure diagnostics (no counterpart in the paper), readable while other
 * streams are stuck: copies the device-side records on the library's own
 * non-blocking stream into pinned host memory and polls for up to `wait_ms`.
 *   out[0]    the status word (1 when a bounded wait gave up since the last clear)
 *   out[1..3] GEMM CTAs counted at entry, after set-up and at exit (since load)
 *   out[4..7] the first give-up since the last clear: site code ((epilogue kind
 *             + 1) * 100 + CTA group * 10 + role), CTA index, the barrier's
 *             shared-memory address and the parity waited for; zeros when none
 * The first call creates the stream and the 64-byte pinned buffer; make it while
 * the device is healthy.  TERN_ERR_TIMEOUT when the copies did not finish in time.
 */
int tern_device_diagnostics(int64_t* out, int wait_ms);

/*
 * Self-test of failure detection (no counterpart in the paper): enqueue one
 * kernel that waits, with the GEMMs' bounded-wait routine and a limit of
 * limit_us microseconds (1..2e6), on an mbarrier nothing arrives on.  It gives
 * up, records TERN_ERR_TIMEOUT in the device status word (see
 * tern_device_status) and returns; the context stays usable.
 */
int tern_selftest_wait_timeout(unsigned limit_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TERN_H */
