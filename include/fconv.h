/*
 * fconv.h -- C ABI of the GB300 FusedConv library (libfconv.so).
 *
 * FusedConv computes  Y = act(conv(X, W) + B + Z)  for 1 to 3 spatial dimensions
 * (com.microsoft.FusedConv kernel package, README "Description": an N-d convolution,
 * an optional bias B, an optional residual Z added before the activation, then an
 * optional fused activation; float16 or float32; 1-3 spatial dimensions).
 *
 * Tensor layouts (README "Inputs"/"Outputs"; manifest "inputs"/"outputs"):
 *   X  (N, C, D1..Dn)          contiguous, channels-first (NCW / NCHW / NCDHW)
 *   W  (M, C/group, k1..kn)    contiguous (OIW / OIHW / OIDHW)
 *   B  (M)                     optional
 *   Z  same shape as Y         optional
 *   Y  (N, M, O1..On)          output; shape from fconv_plan_output_shape
 * All five share the element type T (manifest typeConstraints: float32, float16).
 * Device pointers must be 16-byte aligned (what cudaMalloc and PyTorch give).
 *
 * Ownership: the caller owns every tensor and the workspace; a plan owns only host
 * state. Y must not overlap X, W, B, Z or the workspace.
 *
 * Errors: every attribute and shape rule is checked in fconv_plan_create, before
 * anything is allocated or launched; fconv_run checks pointers, alignment and the
 * workspace, then enqueues asynchronously on the given stream. On any error detected
 * on the host nothing is launched and Y is not written. No call aborts the process.
 */
#ifndef FCONV_H_
#define FCONV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type T of X, W, B, Z and Y (manifest "typeConstraints"). */
typedef enum { FCONV_F32 = 0, FCONV_F16 = 1 } fconv_dtype;

/* auto_pad (README "Attributes": NOTSET uses pads; SAME_UPPER / SAME_LOWER pick pads so
 * each output size is ceil(input / stride), the odd pixel at the end / the beginning;
 * VALID pads nothing). Manifest derive: samePad*, samePadFront/Top/Left. */
typedef enum {
  FCONV_PAD_NOTSET = 0,
  FCONV_PAD_SAME_UPPER = 1,
  FCONV_PAD_SAME_LOWER = 2,
  FCONV_PAD_VALID = 3
} fconv_autopad;

/* Fused activations, in the order of the manifest's attributeConstraints list.
 * Parameters (README "activation_params"; manifest derive actAlpha/actBeta):
 *   LEAKYRELU       exactly [alpha]
 *   HARDSIGMOID     exactly [alpha, beta]     max(0, min(1, alpha*v + beta))
 *   CLIP            exactly [min, max]
 *   QUICKGELU       optional [alpha] = 1.702  v * sigmoid(alpha*v)
 *   ELU             optional [alpha] = 1.0
 *   THRESHOLDEDRELU optional [alpha] = 1.0    v > alpha ? v : 0
 *   GELU            optional [approximate] = 0 (0: erf form, nonzero: tanh form)
 *   all others      parameters ignored (FASTGELU is always the tanh form). */
typedef enum {
  FCONV_ACT_NONE = 0,
  FCONV_ACT_RELU = 1,
  FCONV_ACT_LEAKYRELU = 2,
  FCONV_ACT_SIGMOID = 3,
  FCONV_ACT_TANH = 4,
  FCONV_ACT_HARDSIGMOID = 5,
  FCONV_ACT_HARDSWISH = 6,
  FCONV_ACT_CLIP = 7,
  FCONV_ACT_QUICKGELU = 8,
  FCONV_ACT_ELU = 9,
  FCONV_ACT_GELU = 10,
  FCONV_ACT_FASTGELU = 11,
  FCONV_ACT_SOFTPLUS = 12,
  FCONV_ACT_THRESHOLDEDRELU = 13,
  FCONV_ACT_ERF = 14
} fconv_act;

typedef enum {
  FCONV_OK = 0,
  FCONV_E_NULL = 1,              /* a required pointer argument is NULL */
  FCONV_E_RANK = 2,              /* X/W rank not 3..5, ranks differ, or a zero extent */
  FCONV_E_ATTR_LENGTH = 3,       /* kernel_shape/strides/dilations need spatialRank entries,
                                    pads 2*spatialRank (manifest *LengthOk) */
  FCONV_E_ATTR_VALUE = 4,        /* stride/dilation < 1, pad < 0, kernel extent < 1 */
  FCONV_E_PADS_WITH_AUTOPAD = 5, /* pads given with auto_pad != NOTSET (explicitPadsOk) */
  FCONV_E_KERNEL_SHAPE = 6,      /* kernel_shape differs from W (kernelShapeMatchesWeights) */
  FCONV_E_GROUP = 7,             /* group < 1, M % group != 0 or W.dim1 * group != C (groupOk) */
  FCONV_E_BIAS_SHAPE = 8,        /* bias length != M (biasOk) */
  FCONV_E_Z_SHAPE = 9,           /* Z shape != Y shape (zOk) */
  FCONV_E_ACT_PARAMS = 10,       /* activation_params count not allowed (activationParamsOk) */
  FCONV_E_ACTIVATION = 11,       /* unknown activation id */
  FCONV_E_OUTPUT_EMPTY = 12,     /* some output extent < 1 */
  FCONV_E_WORKSPACE = 13,        /* workspace smaller than fconv_plan_workspace_size */
  FCONV_E_UNSUPPORTED = 14,      /* valid request this library does not run (e.g. dtype) */
  FCONV_E_CUDA = 15,             /* a CUDA runtime call or launch failed */
  FCONV_E_DEVICE_TIMEOUT = 16,   /* a kernel gave up a bounded wait (device error word) */
  FCONV_E_NOMEM = 17,            /* host allocation failed */
  FCONV_E_ALIGNMENT = 18,        /* a device pointer is not 16-byte aligned */
  FCONV_E_ALIAS = 19             /* Y equals X, W, B, Z or the workspace */
} fconv_status;

/* Kernel routes a plan can take. */
typedef enum {
  FCONV_ROUTE_AUTO = 0,     /* the planner chooses */
  FCONV_ROUTE_DIRECT = 1,   /* CUDA-core direct convolution: every dtype, rank, group */
  FCONV_ROUTE_IGEMM_TC = 2, /* tcgen05 implicit GEMM (float16): in-kernel im2col gather to
                               shared memory, accumulator in tensor memory, fused epilogue */
  FCONV_ROUTE_DEPTHWISE = 3, /* CUDA-core depthwise 2-D kernel (C == M == group) */
  FCONV_ROUTE_GROUPED = 4,   /* CUDA-core grouped conv with small groups (C/group <= 16,
                                M/group <= 32), any rank: shared-memory halo box per (image,
                                group, output box), f32 accumulation. The planner picks it
                                when also C/group * prod(kernel) <= 64. */
  FCONV_ROUTE_TRANSPOSED = 5 /* CUDA-core transposed conv in gather form (desc.transposed):
                                a warp takes 32 outputs of one stride phase, so its lanes
                                share the valid taps; any rank and group, f32 accumulation */
} fconv_route;

/* Operator inputs and attributes (manifest "inputs", "attributes"; README "Attributes").
 * Only the first `rank` entries of x_shape/w_shape and the first spatialRank
 * (= rank - 2) entries of kernel_shape/strides/dilations are read; pads holds
 * [begin_axis0.., end_axis0..]. A count of 0 means the attribute is absent
 * (defaults: strides 1, dilations 1, pads 0, kernel_shape from W). */
typedef struct {
  fconv_dtype dtype;
  int rank;                     /* rank of X and W: 3, 4 or 5 */
  int64_t x_shape[5];
  int64_t w_shape[5];
  int has_bias;                 /* B present; its length must be bias_len == M */
  int64_t bias_len;
  int has_z;                    /* Z present; its shape must equal Y's */
  int z_rank;
  int64_t z_shape[5];
  int64_t group;                /* >= 1 (default 1) */
  fconv_autopad auto_pad;
  int n_kernel_shape, n_strides, n_dilations, n_pads;
  int64_t kernel_shape[3], strides[3], dilations[3], pads[6];
  fconv_act activation;
  int n_act_params;             /* -1: attribute absent; else 0..2 values given */
  float act_params[2];
  /* Transposed convolution (ExecuTorch WebGPU PR #20849, the transposed form of
   * aten.convolution.default): Y = act(convT(X, W) + B + Z) where input position i adds
   * X[n, c, i] * W[c, m, k] to output position i*stride - pad_begin + k*dilation. W is then
   * (C, M/group, kernel...), M = W.dim1 * group, and per axis
   *   out = (in - 1)*stride - pad_begin - pad_end + dilation*(k - 1) + output_padding + 1
   * with 0 <= output_padding < stride. auto_pad must be NOTSET or VALID. With transposed = 0
   * output_padding must be absent or all zero. Zero-initialised descriptors are direct
   * convolutions. */
  int transposed;
  int n_output_padding;         /* 0 = absent; else spatialRank values */
  int64_t output_padding[3];
} fconv_desc;

/* Arithmetic modes. FCONV_PRECISION_HALF2_ROWS (opt-in, f16 2-D depthwise convs on the
 * tiled depthwise kernel only; other requests return FCONV_E_UNSUPPORTED): the taps of each
 * kernel row are summed for two adjacent outputs with packed f16 FMAs (each rounded once to
 * f16) and the row partials are added in f32. Its error is bounded by the f16 output
 * rounding plus K * 2^-11 * sum|x*w| (K taps per row), outside the default f16 tolerance
 * (2e-3*|ref| + 1e-3*sum|x*w|/sqrt(Kg)); it takes fewer instructions per output. */
typedef enum {
  FCONV_PRECISION_DEFAULT = 0,
  FCONV_PRECISION_HALF2_ROWS = 1
} fconv_precision;

/* Planner overrides, for tests and experiments. Zero-initialise for defaults. */
typedef struct {
  fconv_route route;            /* FCONV_ROUTE_AUTO = choose */
  int split_k;                  /* 0 = choose; >= 1 forces that many K splits (IGEMM_TC) */
  int tile_n;                   /* 0 = choose; else the largest pixel tile (MMA N) of the
                                   tensor-core kernels: 64, 128 or 256 (their channel tiles
                                   are 128) */
  int a_path;                   /* IGEMM_TC A operand: 0 = choose, 1 = in-kernel gather from
                                   X, 2 = TMA boxes of X repacked in 64-channel blocks (needs
                                   C/group % 64 == 0 and strides <= 8) */
  int max_ctas;                 /* 0 = as many persistent CTAs as the work and the SMs allow;
                                   else at most this many (the persistent kernels then walk
                                   more work units per CTA) */
  int precision;                /* fconv_precision (0 = the default: f32 accumulation) */
} fconv_options;

typedef struct fconv_plan fconv_plan;

/* Validate the request and build a plan: shapes (manifest derive expectedOutput*),
 * applied pads (effectivePad*, samePad*), route, tile and split-K factor. `device` is
 * the CUDA ordinal whose SM count the heuristics use (-1: the current device; with no
 * device present the plan assumes 152 SMs). Returns FCONV_OK and *out, or an error and
 * *out = NULL. */
fconv_status fconv_plan_create(const fconv_desc* desc, int device, fconv_plan** out);

/* As fconv_plan_create, with planner overrides (NULL = defaults). A forced route that
 * cannot run the request returns FCONV_E_UNSUPPORTED. */
fconv_status fconv_plan_create_ex(const fconv_desc* desc, int device,
                                  const fconv_options* opts, fconv_plan** out);

/* Y's shape (rank entries, rank = X's rank). */
fconv_status fconv_plan_output_shape(const fconv_plan* plan, int64_t y_shape[5], int* rank);

/* Applied begin/end pads per (depth, height, width) axis; missing axes read 0. */
fconv_status fconv_plan_pads(const fconv_plan* plan, int64_t pad_begin[3], int64_t pad_end[3]);

/* Device workspace bytes fconv_run needs. On the tensor-core route: the weights copied
 * into the GEMM's K order (unless W is already in it), X repacked with channels innermost
 * for the A operand, and the f32 partial sums of a split-K plan; 0 on the direct and
 * depthwise routes. */
fconv_status fconv_plan_workspace_size(const fconv_plan* plan, size_t* bytes);

/* Route, tile and split chosen by the plan. */
fconv_status fconv_plan_route(const fconv_plan* plan, fconv_route* route, int* tile_n,
                              int* split_k);

/* Number of kernels one fconv_run of this plan launches: one on the direct and depthwise
 * routes; on the tensor-core route a prologue (weight copy and X repack in one launch),
 * the implicit GEMM and, when K is split, the reduction of the partial sums. */
fconv_status fconv_plan_launches(const fconv_plan* plan, int* kernels);

/* Algorithmic work of one fconv_run: 2 * N * P * M * (C/group) * prod(kernel) flops and
 * the bytes of X, W, B, Z and Y each counted once. */
fconv_status fconv_plan_work(const fconv_plan* plan, double* flops, double* bytes);

/* Enqueue Y = act(conv(X, W) + B + Z) on `stream` (a cudaStream_t; NULL = legacy default).
 * x, w, y: device pointers; b, z: device pointers or NULL (must match has_bias/has_z);
 * workspace: device memory of at least fconv_plan_workspace_size bytes (may be NULL when
 * that is 0). Asynchronous: returns after the launch; kernel faults surface on the next
 * synchronising CUDA call. */
fconv_status fconv_run(const fconv_plan* plan, const void* x, const void* w, const void* b,
                       const void* z, void* y, void* workspace, size_t workspace_bytes,
                       void* stream);

/* Synchronise `stream`, then read and clear the device error word that kernels set when
 * a bounded wait gives up. FCONV_OK, FCONV_E_DEVICE_TIMEOUT or FCONV_E_CUDA. */
fconv_status fconv_check_device(void* stream);

/* fconv_run for callers that cannot allocate device memory: code running where
 * cudaMalloc is unavailable or forbidden (inside a capture or allocator hook that must
 * not allocate, a host callback, a plugin whose host application owns every device
 * allocation, or a real-time path with a no-allocation rule). It takes the same
 * arguments as fconv_run minus the workspace: the workspace the plan needs
 * (fconv_plan_workspace_size: the weight copy, the repacked X and any split-K partial
 * sums of the tensor-core route) comes from a fixed array of FCONV_NOALLOC_SCRATCH_BYTES
 * compiled into the library, which every GPU that loads the library keeps until the
 * process exits. The pages this library follows have no counterpart of this call.
 *  - A plan needing more scratch than FCONV_NOALLOC_SCRATCH_BYTES is rejected with
 *    FCONV_E_WORKSPACE before anything is launched.
 *  - The device is the current CUDA device; x, w, b, z, y and `stream` must belong to it.
 *    The first call on a device whose plan needs a workspace looks up the array's device
 *    address (cudaGetSymbolAddress) and keeps it; make that first call before any stream
 *    capture. Plans that need no workspace (direct and depthwise routes) never touch the
 *    array. The kept address does not survive cudaDeviceReset: do not use this entry
 *    point again in a process after resetting the device.
 *  - Calls share the one array per device. It keeps the last call's contents; the
 *    kernels overwrite every scratch element they later read, so nothing is cleared.
 *    Calls whose kernels overlap on the GPU (other streams, other host threads) race on
 *    it: serialise them. Nothing here calls cudaMalloc, cudaFree or an allocating
 *    library routine. */
#define FCONV_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
fconv_status fconv_run_noalloc(const fconv_plan* plan, const void* x, const void* w,
                               const void* b, const void* z, void* y, void* stream);

void fconv_destroy(fconv_plan* plan);

const char* fconv_status_string(fconv_status status);

/* Library version as an integer, major * 10000 + minor * 100 + patch. */
int fconv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FCONV_H_ */
