/*
 * forge.h -- C ABI of the fused weight-gradient + optimizer-step library (libforge.so).
 *
 * The method is FORGE ("FORGE: Fused On-Register Gradient Elimination for
 * Memory-Efficient LLM Training", gist.science technical summary).  Its §2
 * Methodology, Core mechanism, processes the weight matrix of a linear layer
 * one 128 x 128 tile at a time: (1) the tile of the weight gradient
 * dW = dY^T X is accumulated in FP32 on chip, (2) the optimizer update is
 * applied to the finished tile on chip, (3) the gradient tile is discarded and
 * never written to device memory, (4) only the updated weight tile and the
 * (optionally quantised) moment tiles are written back.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - The layer is Y = X W^T with W of shape [d_out, d_in].
 *  - dY is [T, d_out] and X is [T, d_in]: bfloat16, row-major (token-major), as
 *    the forward and backward passes of a linear layer leave them.
 *  - W is [d_out, d_in] bfloat16, row-major.  m and v are [d_out, d_in] row-major,
 *    binary32 (FORGE_STATE_FP32), int8 codes (FORGE_STATE_INT8_B64) or bfloat16
 *    (FORGE_STATE_BF16).
 *  - BF16 states: the update reads the stored moments as binary32 and computes the
 *    new ones in binary32 (the weight update uses these); they are then stored by
 *    stochastic rounding to bfloat16 with 16 Philox bits each, like the weight,
 *    from separate streams: the high counter word of the weight's stream gains
 *    1 << 30 for m and 2 << 30 for v.
 *  - INT8 states (§2 Precision and fidelity, third low-precision point: blocks
 *    of 64): each run of 64 consecutive elements of a row shares one binary32
 *    scale s = absmax / 127; code q = clamp(round_half_even(x / s), -127, 127);
 *    value = q * s.  `qscales` then points to 2 * d_out * d_in / 64 binary32
 *    scales: the m scales first ([d_out, d_in/64] row-major), then the v scales.
 *  - All pointers are DEVICE pointers of the current CUDA device, owned by the
 *    caller.  The library allocates no device memory and keeps no pointer after a
 *    call returns.  W, m, v and qscales are updated in place.
 *  - Alignment: every tensor pointer (dY, X, W, m, v, dW, dX) must be 32-byte
 *    aligned, qscales 4-byte aligned, per-channel scale vectors 16-byte aligned.
 *    TMA would accept 16-byte aligned dY and X; the stricter rule is the
 *    epilogue's: it reads and writes W, m, v, dW and dX with 256-bit accesses
 *    (8 binary32 moments or 16 bfloat16 values per instruction), which need
 *    32-byte aligned addresses, and a pointer that fails it is rejected with
 *    FORGE_ERR_MISALIGNED before anything is launched.
 *  - Sizes: d_out and d_in multiples of 8 (a TMA row stride is a multiple of 16
 *    bytes; with INT8 states d_in is a multiple of 64, so that a block of 64
 *    never spans two rows) and any T >= 0.  The method's 128 x 128 tile (§2
 *    Methodology) need not divide the layer: a tile reaching past the last row,
 *    column or token computes on zero fill and writes nothing outside the layer.
 *    T == 0 is a zero gradient; d_out or d_in == 0 is an empty layer and a no-op.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *    default stream) and return after the launch is queued.  Argument errors
 *    are detected on the host before anything is launched and are returned
 *    synchronously; nothing is written in that case.
 *  - Every on-device wait in the kernels is bounded in time.  A wait that runs
 *    out sets a device status word and the kernel returns early; the word is
 *    read and cleared by forge_sync_status().  There is one status word per
 *    device, shared by every stream: a timeout in a kernel on stream B is
 *    reported by the next forge_sync_status() of any stream of that device, and
 *    that call clears it.
 *  - Ordering (§5 Significance and claims, limitations: the input gradient must
 *    be read before the weights are updated): the layer's input gradient
 *    dX = dY W needs the old W, so it must be enqueued before forge_fused_dw_step
 *    on the same stream.  forge_dx_gemm computes it; forge_linear_backward
 *    enqueues both in that order.
 */
#ifndef FORGE_H_
#define FORGE_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t is `struct CUstream_st *` */

#if defined(__GNUC__)
#define FORGE_API __attribute__((visibility("default")))
#else
#define FORGE_API
#endif

typedef enum forge_status {
    FORGE_OK = 0,
    FORGE_ERR_INVALID_ARGUMENT = 1, /* null pointer, bad size, bad enum, step < 1 */
    FORGE_ERR_UNSUPPORTED = 2,      /* valid but not implemented (e.g. INT8 states for SGD) */
    FORGE_ERR_MISALIGNED = 3,       /* a pointer is not 32-byte aligned */
    FORGE_ERR_CUDA = 4,             /* a CUDA runtime/driver call failed */
    FORGE_ERR_NOT_SM103 = 5,        /* current device is not compute capability 10.3 */
    FORGE_ERR_TIMEOUT = 6           /* a bounded on-device wait ran out (from forge_sync_status) */
} forge_status;

/* The eight element-wise optimizers of §3 Key contributions, "Generality". */
typedef enum forge_opt_kind {
    FORGE_ADAMW = 0,        /* m, v; weight decay decoupled: W <- W (1 - lr wd) */
    FORGE_NADAM = 1,        /* m, v; weight decay coupled:   g <- g + wd W       */
    FORGE_RADAM = 2,        /* m, v; coupled */
    FORGE_LION = 3,         /* m;    decoupled */
    FORGE_RMSPROP = 4,      /* v;    coupled */
    FORGE_ADAGRAD = 5,      /* v;    coupled */
    FORGE_SGD = 6,          /* none; coupled */
    FORGE_SGD_MOMENTUM = 7  /* m;    coupled; m <- momentum m + g (no dampening, not Nesterov) */
} forge_opt_kind;

typedef enum forge_state_dtype {
    FORGE_STATE_FP32 = 0,
    FORGE_STATE_INT8_B64 = 1,
    FORGE_STATE_BF16 = 2  /* §2 Precision and fidelity, "BF16 or INT8" states: see below */
} forge_state_dtype;

typedef struct forge_shape {
    int64_t T;      /* tokens: the contraction length of dW = dY^T X */
    int64_t d_out;  /* rows of W */
    int64_t d_in;   /* columns of W */
    int32_t state;  /* a forge_state_dtype */
    int32_t reserved; /* must be 0 */
} forge_shape;

/* Hyperparameters, each a binary32.  Fields an optimizer does not use are ignored.
 * Step-dependent factors (bias corrections, the NAdam momentum product, the RAdam
 * rectification) are derived on the host in binary64 from these and `step`,
 * assuming the run started at step 1 with the same hyperparameters. */
typedef struct forge_hparams {
    float lr;
    float beta1;          /* Adam-family / Lion first coefficient */
    float beta2;          /* Adam-family second moment / Lion moment coefficient */
    float eps;
    float weight_decay;
    float momentum;       /* SGD-momentum */
    float alpha;          /* RMSprop smoothing constant */
    float momentum_decay; /* NAdam psi */
    float lr_decay;       /* AdaGrad */
} forge_hparams;

/*
 * forge_fused_dw_step -- one fused step for one linear layer (§2 Methodology,
 * Core mechanism, steps 1-4).
 *
 *   For every 128 x 128 tile of W: g = sum_t dY[t, rows]^T X[t, cols] in FP32 on
 *   chip (never written to device memory); the optimizer `opt_kind` updates the
 *   tile's W, m, v with g; the new moments are stored as binary32 or requantised
 *   to INT8 (the update itself uses the unquantised new moments); the new weight,
 *   computed in binary32, is stored as bfloat16 by stochastic rounding (§2
 *   Precision and fidelity, second low-precision point) with 16 bits of a
 *   Philox4x32-10 stream: key (seed mod 2^32, seed div 2^32), counter
 *   (e div 8 as 64 bits, step as 64 bits) for row-major element index e, element
 *   e taking the low (e even) or high (e odd) half of output word (e div 2) mod 4.
 *
 *   m: required for ADAMW, NADAM, RADAM, LION, SGD_MOMENTUM; ignored otherwise.
 *   v: required for ADAMW, NADAM, RADAM, RMSPROP, ADAGRAD; ignored otherwise.
 *   qscales: required iff shape->state == FORGE_STATE_INT8_B64.  SGD has no
 *   states: it takes FORGE_STATE_FP32 only.
 *   step: the 1-based optimizer step t.  seed: the layer's SR seed.
 *   T == 0 applies the update with a zero gradient.
 */
FORGE_API forge_status forge_fused_dw_step(const void *dY, const void *X, void *W, void *m, void *v,
                                 float *qscales, forge_opt_kind opt_kind,
                                 const forge_hparams *hp, const forge_shape *shape,
                                 int64_t step, uint64_t seed, struct CUstream_st *stream);

/* One layer of forge_fused_dw_step_layers: what forge_fused_dw_step takes for it. */
typedef struct forge_layer {
    const void *dY;   /* [T, d_out] bfloat16 */
    const void *X;    /* [T, d_in] bfloat16 */
    void *W;          /* [d_out, d_in] bfloat16, updated in place */
    void *m;          /* moments as for forge_fused_dw_step (NULL where the optimizer keeps none) */
    void *v;
    float *qscales;   /* INT8 states: 2 * d_out * d_in / 64 scales; NULL otherwise */
    int64_t T, d_out, d_in;
    uint64_t seed;    /* the layer's stochastic-rounding seed */
} forge_layer;

/*
 * forge_fused_dw_step_layers -- forge_fused_dw_step for several independent layers at once
 * (§2 Methodology, Core mechanism, applied to every layer of a backward pass; the tile kernel's
 * persistent loop, §4's removal of the separate optimizer launch, extended across layers).
 *
 *   The result is bit for bit that of calling forge_fused_dw_step on each layer in turn with the
 *   same opt_kind, hp, step and state (every element's update and Philox counter depend only on its
 *   own layer).  Layers whose preferred tile is a CTA pair (d_out and d_in multiples of 256, or
 *   ragged above 1024) run together: their tiles are numbered layer after layer and visited by one
 *   persistent schedule, up to 16 layers per launch, so the pipeline fills and drains once per
 *   launch instead of once per layer.  Other layers (and layers with T == 0) are launched one by
 *   one, as forge_fused_dw_step would.
 *
 *   layers: n_layers entries, host memory, read during the call only.  The layers must be
 *   independent: no layer's W, m, v or qscales may overlap any other buffer of any layer.
 *   state: a forge_state_dtype, the same for every layer.  bf16 operands only (the E4M3 entry
 *   points take one layer per call).  Every layer is checked as forge_fused_dw_step checks its
 *   arguments before anything is launched; an error names no layer and launches nothing.
 */
FORGE_API forge_status forge_fused_dw_step_layers(const forge_layer *layers, int32_t n_layers, int32_t state,
                                                  forge_opt_kind opt_kind, const forge_hparams *hp, int64_t step,
                                                  struct CUstream_st *stream);

/*
 * forge_dw_gemm -- the weight gradient alone, written to device memory: dW [d_out,
 * d_in] binary32 row-major, dW = dY^T X accumulated in FP32.  This is the first
 * half of the two-phase schedule of §1 The problem (backward writes the full
 * gradient, the optimizer reads it back); it exists only as the unfused
 * baseline.  shape->state is ignored.
 */
FORGE_API forge_status forge_dw_gemm(const void *dY, const void *X, float *dW, const forge_shape *shape,
                           struct CUstream_st *stream);

/*
 * forge_opt_step -- the optimizer half of the two-phase schedule: reads a
 * materialised gradient dW [d_out, d_in] binary32 and applies exactly the update,
 * state write-back and stochastic rounding of forge_fused_dw_step.  shape->T is
 * ignored.  dW == NULL means a zero gradient.
 */
FORGE_API forge_status forge_opt_step(const float *dW, void *W, void *m, void *v, float *qscales,
                            forge_opt_kind opt_kind, const forge_hparams *hp,
                            const forge_shape *shape, int64_t step, uint64_t seed,
                            struct CUstream_st *stream);

/*
 * forge_fused_dw_step_e4m3 -- forge_fused_dw_step with FP8 operands (§4 Experimental
 * results, "Composability": FORGE composes with FP8 quantisation and absorbs the
 * dequantisation cost).  dY [T, d_out] and X [T, d_in] are E4M3 codes (OCP 8-bit
 * format: 4 exponent bits, bias 7, 3 mantissa bits, no infinities), row-major, one
 * byte each, with one binary32 scale per tensor: value = scale * decode(code).  The
 * tensor core sums the code products in FP32 (kind::f8f6f4); the finished gradient
 * tile is then multiplied by s = dy_scale * x_scale (one binary32 product, formed
 * on the host) and the step proceeds exactly as in forge_fused_dw_step, for every
 * state format.  d_out and d_in must be multiples of 16 (row strides of 16 bytes);
 * both scales finite and positive.
 */
FORGE_API forge_status forge_fused_dw_step_e4m3(const void *dY, const void *X, float dy_scale, float x_scale,
                                                void *W, void *m, void *v, float *qscales, forge_opt_kind opt_kind,
                                                const forge_hparams *hp, const forge_shape *shape, int64_t step,
                                                uint64_t seed, struct CUstream_st *stream);

/* The weight gradient alone from E4M3 operands: dW = s * (dY^T X) in binary32, as
 * forge_dw_gemm; the unfused baseline of forge_fused_dw_step_e4m3. */
FORGE_API forge_status forge_dw_gemm_e4m3(const void *dY, const void *X, float dy_scale, float x_scale, float *dW,
                                          const forge_shape *shape, struct CUstream_st *stream);

/*
 * forge_fused_dw_step_e4m3_channels, forge_dw_gemm_e4m3_channels -- the same with one scale
 * per channel: dy_scales [d_out] (one per column of dY, the output channels) and x_scales
 * [d_in] (one per column of X), binary32 device vectors, 16-byte aligned, read-only.  They
 * factor out of the sum over tokens like the per-tensor scales, so each gradient element is
 * multiplied by its own binary32 product dy_scales[o] * x_scales[i], formed in the epilogue.
 * Per-tensor scaling is the case of constant vectors (and gives identical results).
 */
FORGE_API forge_status forge_fused_dw_step_e4m3_channels(const void *dY, const void *X, const float *dy_scales,
                                                         const float *x_scales, void *W, void *m, void *v,
                                                         float *qscales, forge_opt_kind opt_kind,
                                                         const forge_hparams *hp, const forge_shape *shape,
                                                         int64_t step, uint64_t seed, struct CUstream_st *stream);

FORGE_API forge_status forge_dw_gemm_e4m3_channels(const void *dY, const void *X, const float *dy_scales,
                                                   const float *x_scales, float *dW, const forge_shape *shape,
                                                   struct CUstream_st *stream);

/*
 * forge_dx_gemm -- the layer's input gradient dX = dY W (the read of W that §5
 * Significance and claims, limitations, requires before the update), on the
 * tensor cores: dX[t, i] = sum_o dY[t, o] W[o, i], accumulated in FP32 on chip
 * and stored once, rounded to nearest even, as bfloat16.
 *
 *   dY [T, d_out] and W [d_out, d_in] bfloat16 row-major, as for the fused step;
 *   dX [T, d_in] bfloat16 row-major, written (not accumulated); it must not
 *   overlap dY or W.  Any T >= 0 is accepted (a tail of fewer than 128 or 256
 *   tokens is computed on zero fill and not stored).  d_out == 0 writes zeros;
 *   T == 0 or d_in == 0 writes nothing.  shape->state is ignored.
 */
FORGE_API forge_status forge_dx_gemm(const void *dY, const void *W, void *dX, const forge_shape *shape,
                                     struct CUstream_st *stream);

/*
 * forge_linear_backward -- the whole backward of the linear layer Y = X W^T with
 * the fused weight step, in the order §5 Significance and claims, limitations,
 * requires: forge_dx_gemm (dX from the weights before the step), then
 * forge_fused_dw_step, both on `stream`.  Arguments are those of the two calls;
 * all of them are checked before either is launched, so an argument error
 * launches nothing.  dX must not overlap any other buffer.
 */
FORGE_API forge_status forge_linear_backward(const void *dY, const void *X, void *W, void *m, void *v,
                                             float *qscales, void *dX, forge_opt_kind opt_kind,
                                             const forge_hparams *hp, const forge_shape *shape, int64_t step,
                                             uint64_t seed, struct CUstream_st *stream);

/* Waits for `stream`, then reads and clears the device status word of the current
 * device: FORGE_ERR_TIMEOUT if a bounded wait ran out in a kernel (on any stream of
 * this device) since the last read, FORGE_ERR_CUDA if the stream reported an error,
 * FORGE_OK otherwise.  A timeout on another stream still running may be reported by a
 * later call. */
FORGE_API forge_status forge_sync_status(struct CUstream_st *stream);

/* Time limit of every bounded on-device wait, in nanoseconds (default 2e9).
 * Values below 1e6 are raised to 1e6.  Host-side setting, applies to later launches.
 * The epilogue's wait for a finished accumulator spans a whole tile mainloop, whose
 * length grows with the reduction: it gets the limit plus 4 us per 64-token slice
 * (128 for E4M3 operands; per 64 rows of d_out for forge_dx_gemm), far above the
 * slice's time on a GB300, so that a long but healthy run never reports a timeout. */
FORGE_API void forge_set_wait_limit_ns(uint64_t ns);

/* Test switch for the failure-detection path (the method has no counterpart; it exists so that
 * the bounded waits can be exercised without a real fault).  The next tile-kernel launch (of
 * forge_fused_dw_step, forge_fused_dw_step_e4m3, forge_dw_gemm, forge_dw_gemm_e4m3 or
 * forge_dx_gemm, with work to do) arms the first pipeline stage of its first tile but never copies
 * into it: the MMA thread's wait for that stage runs out after the wait limit, the kernel records
 * FORGE_ERR_TIMEOUT, stops every other wait, waits (bounded) until every copy it did issue into
 * shared memory has landed, frees its TMEM and returns; forge_sync_status() then reports FORGE_ERR_TIMEOUT and the
 * CUDA context stays usable.  The outputs of that one call are unspecified.  No fault is raised. */
FORGE_API void forge_debug_withhold_next_stage(void);

/* The tile shape and persistent grid forge_fused_dw_step (and forge_dw_gemm) use for `shape` with
 * bf16 operands: rows x columns of W per tile (256 x 256 on a CTA pair, a group of the method's
 * 128 x 128 tiles, §2 Methodology; 128 x 256 or 128 x 128 on one CTA; a layer whose wider shape
 * would occupy at most half the SMs takes 128 x 128, and if those would too, 128 x 64 -- half of
 * one of the method's tiles -- except with INT8 states), CTAs per thread-block cluster (1 or 2),
 * and CTAs launched on the current device.  E4M3 operands never take 128 x 64 tiles: where the
 * query answers 128 x 64 they run on 128 x 128.  With bf16 operands, a pair launch whose last wave
 * of 256 x 256 tiles would occupy at most half of the pairs runs those last tiles as two 256 x 128
 * halves each (the query reports the 256 x 256 tile).  Host-side query, no launch; it reads the
 * device's SM count, so it needs a device (FORGE_ERR_CUDA or FORGE_ERR_NOT_SM103 otherwise). */
FORGE_API forge_status forge_launch_shape(const forge_shape *shape, int32_t *tile_rows, int32_t *tile_cols,
                                          int32_t *cluster, int32_t *ctas);

/* The same for forge_dx_gemm: tokens x d_in columns of dX per tile, CTAs per cluster, CTAs. */
FORGE_API forge_status forge_dx_launch_shape(const forge_shape *shape, int32_t *tile_rows, int32_t *tile_cols,
                                             int32_t *cluster, int32_t *ctas);

/* Number of the library's own kernel launches queued since load (all entry points). */
FORGE_API uint64_t forge_launch_count(void);

/* A static, NUL-terminated description of a status code. */
FORGE_API const char *forge_status_string(forge_status status);

#ifdef __cplusplus
}
#endif

#endif /* FORGE_H_ */
