/*
 * FusedConv CPU oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow direct convolution in double precision that defines what the GPU
 * library must compute. Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg load this file's library; the product path never does. It shares
 * no code, header or constant with the CUDA library.
 *
 * Sources (com.microsoft.FusedConv kernel package):
 *  - manifest.json "derive": the spatial extents (inputDepth/Height/Width,
 *    kernelDepth/Height/Width), the attribute reads (kernelD.., strideD.., dilationD..,
 *    padFront..padRight), the SAME padding split (samePad*, samePadFront/Top/Left),
 *    the effective begin pads (effectivePad*), the expected output sizes
 *    (expectedOutputDepth/Height/Width), the validation predicates
 *    (kernelShapeLengthOk ... explicitPadsOk, spatialAttributesOk, groupOk, biasOk, zOk,
 *    activationParamsOk) and the activation parameter defaults (actAlpha, actBeta).
 *  - README.md "Description", "Inputs", "Attributes": Y = act(conv(X, W) + B + Z),
 *    Z is added before the activation, the activation list and activation_params.
 *  - The index mapping of a padded, strided, dilated tap (input = out*stride - pad_begin
 *    + tap*dilation, zero outside the input) is the one the ExecuTorch conv2d_gemm PR
 *    (#20873, "on-the-fly sampling ... zero when out of range") and the manifest's
 *    params_ncdhw3d block (padD/padH/padW = effectivePad*) describe.
 *
 * Transposed convolution (oracle_conv_transpose): ExecuTorch WebGPU PR #20849, the
 * transposed form of aten.convolution.default ("conv_transpose2d.wgsl ... gather-form
 * transposed conv", weight "in the un-flipped torch transposed layout [IC, OC/groups, KH,
 * KW]", "output_padding >= stride" rejected). The oracle writes the definition in its
 * scatter form: every input element adds x * w to the output at
 * input*stride - pad_begin + tap*dilation.
 *
 * Parity is pinned by the tests against PyTorch CPU float64 convolutions (a library
 * routine), brute force on tiny inputs, 1x1 conv == matmul, the delta kernel,
 * rank embedding, closed-form activation values and the output-size formulas; the
 * transposed convolution additionally by the adjoint identity with the (pinned) direct
 * convolution and by closed forms on tiny inputs.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Status codes of the oracle (independent of the CUDA library's codes). */
enum {
  OR_OK = 0,
  OR_BAD_RANK = 1,        /* x/w rank not 3..5 or not equal */
  OR_ATTR_LENGTH = 2,     /* kernel_shape/strides/dilations/pads length mismatch */
  OR_ATTR_VALUE = 3,      /* stride/dilation < 1, pad < 0, kernel extent < 1 */
  OR_PADS_AUTOPAD = 4,    /* explicit pads with auto_pad != NOTSET */
  OR_KERNEL_SHAPE = 5,    /* kernel_shape does not match W */
  OR_GROUP = 6,           /* group < 1, M % group != 0, W.dim1 * group != C */
  OR_ACT_PARAMS = 7,      /* activation_params count not allowed for the activation */
  OR_ACTIVATION = 8,      /* unknown activation */
  OR_EMPTY_OUTPUT = 9,    /* an output extent < 1 */
  OR_NULL = 10
};

/* Activation ids, in the order of the manifest's attributeConstraints list; 0 = none. */
enum {
  A_NONE = 0, A_RELU, A_LEAKYRELU, A_SIGMOID, A_TANH, A_HARDSIGMOID, A_HARDSWISH, A_CLIP,
  A_QUICKGELU, A_ELU, A_GELU, A_FASTGELU, A_SOFTPLUS, A_THRESHOLDEDRELU, A_ERF, A_COUNT
};

/* auto_pad modes */
enum { P_NOTSET = 0, P_SAME_UPPER = 1, P_SAME_LOWER = 2, P_VALID = 3 };

typedef struct {
  int rank;                    /* rank of X and W: 3, 4 or 5 */
  int64_t x_shape[5];
  int64_t w_shape[5];
  int64_t group;
  int auto_pad;
  int n_kernel_shape, n_strides, n_dilations, n_pads;   /* 0 = attribute absent */
  int64_t kernel_shape[3], strides[3], dilations[3], pads[6];
  int activation;
  int n_act_params;            /* -1 = attribute absent */
  double act_params[2];
} oracle_attrs;

typedef struct {
  int spatial_rank;
  int64_t in[3], k[3], s[3], d[3];   /* depth, height, width (1 for missing axes) */
  int64_t pad_begin[3], pad_end[3];  /* the padding actually applied */
  int64_t out[3];
  int64_t N, C, M, G, Cg, Mg;
  double alpha, beta;
} oracle_geom;

/* floor(a / b) for b > 0 and any sign of a */
static int64_t floordiv(int64_t a, int64_t b) {
  int64_t q = a / b;
  if ((a % b != 0) && (a < 0)) q -= 1;
  return q;
}

/*
 * Resolve attributes into the geometry, following the manifest's derive block axis by
 * axis. Axis j of the (depth, height, width) triple takes attribute index
 * j - (3 - spatialRank); axes that the rank does not have are 1 (sizes, kernel,
 * stride, dilation) or 0 (pads).
 */
int oracle_resolve(const oracle_attrs* a, oracle_geom* g) {
  if (!a || !g) return OR_NULL;
  memset(g, 0, sizeof(*g));
  if (a->rank < 3 || a->rank > 5) return OR_BAD_RANK;
  const int sr = a->rank - 2;
  g->spatial_rank = sr;
  /* lengths (kernelShapeLengthOk, stridesLengthOk, dilationsLengthOk, padsLengthOk) */
  if (a->n_kernel_shape && a->n_kernel_shape != sr) return OR_ATTR_LENGTH;
  if (a->n_strides && a->n_strides != sr) return OR_ATTR_LENGTH;
  if (a->n_dilations && a->n_dilations != sr) return OR_ATTR_LENGTH;
  if (a->n_pads && a->n_pads != 2 * sr) return OR_ATTR_LENGTH;
  for (int j = 0; j < 3; ++j) {
    int ax = j - (3 - sr);               /* attribute index, < 0 if the axis is absent */
    if (ax < 0) {
      g->in[j] = 1; g->k[j] = 1; g->s[j] = 1; g->d[j] = 1;
      g->pad_begin[j] = 0; g->pad_end[j] = 0;
      continue;
    }
    g->in[j] = a->x_shape[2 + ax];
    g->k[j] = a->w_shape[2 + ax];
    g->s[j] = a->n_strides ? a->strides[ax] : 1;
    g->d[j] = a->n_dilations ? a->dilations[ax] : 1;
    g->pad_begin[j] = a->n_pads ? a->pads[ax] : 0;
    g->pad_end[j] = a->n_pads ? a->pads[sr + ax] : 0;
    /* kernelShapeMatchesWeights */
    if (a->n_kernel_shape && a->kernel_shape[ax] != g->k[j]) return OR_KERNEL_SHAPE;
  }
  for (int j = 0; j < 3; ++j) {
    if (g->k[j] < 1) return OR_ATTR_VALUE;                       /* kernelExtentsOk */
    if (g->s[j] < 1 || g->d[j] < 1) return OR_ATTR_VALUE;        /* strides/dilationsValuesOk */
    if (g->pad_begin[j] < 0 || g->pad_end[j] < 0) return OR_ATTR_VALUE;  /* padsValuesOk */
  }
  /* explicitPadsOk: explicit pads only with NOTSET */
  if (a->auto_pad != P_NOTSET && a->n_pads) return OR_PADS_AUTOPAD;
  if (a->auto_pad < P_NOTSET || a->auto_pad > P_VALID) return OR_ATTR_VALUE;

  for (int j = 0; j < 3; ++j) {
    const int64_t in = g->in[j], k = g->k[j], s = g->s[j], d = g->d[j];
    const int64_t ext = (k - 1) * d + 1;
    if (a->auto_pad == P_SAME_UPPER || a->auto_pad == P_SAME_LOWER) {
      /* expectedOutput*: ceil(in / stride); samePad*: the total; samePadFront/Top/Left */
      int64_t out = (in + s - 1) / s;
      int64_t total = (out - 1) * s + ext - in;
      if (total < 0) total = 0;
      int64_t half = total / 2;
      g->pad_begin[j] = (a->auto_pad == P_SAME_UPPER) ? half : total - half;
      g->pad_end[j] = total - g->pad_begin[j];
      g->out[j] = out;
    } else {
      if (a->auto_pad == P_VALID) { g->pad_begin[j] = 0; g->pad_end[j] = 0; }
      /* floor((in + pads - ((k - 1) * d + 1)) / stride) + 1 */
      g->out[j] = floordiv(in + g->pad_begin[j] + g->pad_end[j] - ext, s) + 1;
    }
    if (g->out[j] < 1) return OR_EMPTY_OUTPUT;
  }
  /* groupOk */
  g->N = a->x_shape[0];
  g->C = a->x_shape[1];
  g->M = a->w_shape[0];
  g->G = a->group;
  if (g->G < 1 || g->M % g->G != 0 || a->w_shape[1] * g->G != g->C) return OR_GROUP;
  g->Cg = a->w_shape[1];
  g->Mg = g->M / g->G;
  if (g->N < 1 || g->C < 1 || g->M < 1) return OR_BAD_RANK;

  /* activationOk and activationParamsOk; defaults from actAlpha / actBeta */
  const int act = a->activation, np = a->n_act_params;
  if (act < 0 || act >= A_COUNT) return OR_ACTIVATION;
  if (act == A_LEAKYRELU && np != 1) return OR_ACT_PARAMS;
  if ((act == A_HARDSIGMOID || act == A_CLIP) && np != 2) return OR_ACT_PARAMS;
  if ((act == A_QUICKGELU || act == A_ELU || act == A_THRESHOLDEDRELU || act == A_GELU) && np > 1)
    return OR_ACT_PARAMS;
  double alpha = 0.0, beta = 0.0;
  if (act == A_HARDSIGMOID) { alpha = 0.2; beta = 0.5; }
  else if (act == A_LEAKYRELU) alpha = 0.01;
  else if (act == A_QUICKGELU) alpha = 1.702;
  else if (act == A_ELU || act == A_THRESHOLDEDRELU) alpha = 1.0;
  if (np >= 1) alpha = a->act_params[0];
  if (np >= 2) beta = a->act_params[1];
  g->alpha = alpha;
  g->beta = beta;
  return OR_OK;
}

/*
 * The activation of a pre-activation value v, in double precision. The pages name the
 * activations and their parameters (README "Attributes"); the formulas are the
 * textbook/ONNX definitions of those names:
 *   Relu max(v,0); LeakyRelu v<0 ? alpha*v : v; Sigmoid 1/(1+e^-v); Tanh;
 *   HardSigmoid max(0, min(1, alpha*v + beta)); HardSwish v*max(0, min(1, v/6 + 1/2));
 *   Clip min(max(v, lo), hi); QuickGelu v*sigmoid(alpha*v); Elu v>0 ? v : alpha*(e^v - 1);
 *   Gelu 0.5*v*(1 + erf(v/sqrt 2)) or, with the approximate flag, the tanh form;
 *   FastGelu the tanh form; Softplus log(1 + e^v); ThresholdedRelu v>alpha ? v : 0; Erf.
 */
double oracle_activation(int act, double v, double alpha, double beta) {
  const double k_tanh = 0.7978845608028654; /* sqrt(2/pi) */
  switch (act) {
    case A_NONE: return v;
    case A_RELU: return v > 0.0 ? v : 0.0;
    case A_LEAKYRELU: return v < 0.0 ? alpha * v : v;
    case A_SIGMOID: return 1.0 / (1.0 + exp(-v));
    case A_TANH: return tanh(v);
    case A_HARDSIGMOID: {
      double t = alpha * v + beta;
      return t < 0.0 ? 0.0 : (t > 1.0 ? 1.0 : t);
    }
    case A_HARDSWISH: {
      double t = v / 6.0 + 0.5;
      t = t < 0.0 ? 0.0 : (t > 1.0 ? 1.0 : t);
      return v * t;
    }
    case A_CLIP: return v < alpha ? alpha : (v > beta ? beta : v);
    case A_QUICKGELU: return v / (1.0 + exp(-alpha * v));
    case A_ELU: return v > 0.0 ? v : alpha * (exp(v) - 1.0);
    case A_GELU:
      if (alpha != 0.0) return 0.5 * v * (1.0 + tanh(k_tanh * (v + 0.044715 * v * v * v)));
      return 0.5 * v * (1.0 + erf(v / sqrt(2.0)));
    case A_FASTGELU: return 0.5 * v * (1.0 + tanh(k_tanh * (v + 0.044715 * v * v * v)));
    case A_SOFTPLUS: return (v > 0.0 ? v : 0.0) + log1p(exp(-fabs(v)));
    case A_THRESHOLDEDRELU: return v > alpha ? v : 0.0;
    case A_ERF: return erf(v);
    default: return NAN;
  }
}

/* Output shape (rank entries) of a resolved geometry. */
int oracle_output_shape(const oracle_attrs* a, int64_t* y_shape, int64_t* pad_begin,
                        int64_t* pad_end) {
  oracle_geom g;
  int st = oracle_resolve(a, &g);
  if (st != OR_OK) return st;
  y_shape[0] = g.N;
  y_shape[1] = g.M;
  for (int i = 0; i < g.spatial_rank; ++i) y_shape[2 + i] = g.out[3 - g.spatial_rank + i];
  for (int j = 0; j < 3; ++j) {
    if (pad_begin) pad_begin[j] = g.pad_begin[j];
    if (pad_end) pad_end[j] = g.pad_end[j];
  }
  return OR_OK;
}

/*
 * y[n,m,o] = act( sum_{ci<Cg} sum_{tap} x[n, g*Cg+ci, o*s - pad_begin + tap*d] * w[m,ci,tap]
 *                 + b[m] + z[n,m,o] ),  g = m / Mg, x = 0 outside the input.
 * abssum[n,m,o] = sum of |x * w| over the same taps (used for the tolerance).
 * x, w, b, z are double copies of the (already dtype-rounded) tensors; b and z may be NULL.
 * `nthreads` <= 0 uses the OpenMP default.
 */
int oracle_fused_conv(const oracle_attrs* a, const double* x, const double* w, const double* b,
                      const double* z, double* y, double* abssum, int nthreads) {
  oracle_geom g;
  int st = oracle_resolve(a, &g);
  if (st != OR_OK) return st;
  if (!x || !w || !y) return OR_NULL;
  const int64_t ID = g.in[0], IH = g.in[1], IW = g.in[2];
  const int64_t KD = g.k[0], KH = g.k[1], KW = g.k[2];
  const int64_t OD = g.out[0], OH = g.out[1], OW = g.out[2];
  const int64_t P = OD * OH * OW, IS = ID * IH * IW, KS = KD * KH * KW;
  const int64_t NM = g.N * g.M;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int64_t nm = 0; nm < NM; ++nm) {
    const int64_t n = nm / g.M, m = nm % g.M;
    const int64_t grp = m / g.Mg;
    for (int64_t od = 0; od < OD; ++od)
      for (int64_t oh = 0; oh < OH; ++oh)
        for (int64_t ow = 0; ow < OW; ++ow) {
          double acc = 0.0, aacc = 0.0;
          for (int64_t ci = 0; ci < g.Cg; ++ci) {
            const double* xp = x + (n * g.C + grp * g.Cg + ci) * IS;
            const double* wp = w + (m * g.Cg + ci) * KS;
            for (int64_t kz = 0; kz < KD; ++kz) {
              const int64_t iz = od * g.s[0] - g.pad_begin[0] + kz * g.d[0];
              if (iz < 0 || iz >= ID) continue;
              for (int64_t ky = 0; ky < KH; ++ky) {
                const int64_t iy = oh * g.s[1] - g.pad_begin[1] + ky * g.d[1];
                if (iy < 0 || iy >= IH) continue;
                for (int64_t kx = 0; kx < KW; ++kx) {
                  const int64_t ix = ow * g.s[2] - g.pad_begin[2] + kx * g.d[2];
                  if (ix < 0 || ix >= IW) continue;
                  const double p = xp[(iz * IH + iy) * IW + ix] * wp[(kz * KH + ky) * KW + kx];
                  acc += p;
                  aacc += fabs(p);
                }
              }
            }
          }
          const int64_t o = (od * OH + oh) * OW + ow;
          const int64_t yi = (n * g.M + m) * P + o;
          double v = acc;
          if (b) v += b[m];
          if (z) v += z[yi];
          y[yi] = oracle_activation(a->activation, v, g.alpha, g.beta);
          if (abssum) abssum[yi] = aacc;
        }
  }
  return OR_OK;
}

/* ------------------------------------------------------------ transposed convolution */

typedef struct {
  int rank;                    /* rank of X and W: 3, 4 or 5 */
  int64_t x_shape[5];          /* (N, C, spatial...) */
  int64_t w_shape[5];          /* (C, M / group, kernel...) */
  int64_t group;
  int n_strides, n_dilations, n_pads, n_output_padding;  /* 0 = attribute absent */
  int64_t strides[3], dilations[3], pads[6], output_padding[3];
  int activation;
  int n_act_params;            /* -1 = attribute absent */
  double act_params[2];
} oracle_tattrs;

/* Resolve a transposed convolution: per axis
 *   out = (in - 1) * stride - pad_begin - pad_end + dilation * (k - 1) + output_padding + 1
 * with stride, dilation >= 1, pads >= 0 and 0 <= output_padding < stride; C = W.dim0,
 * group divides C, M = W.dim1 * group. The activation rules are those of the direct
 * convolution. */
int oracle_resolve_transpose(const oracle_tattrs* a, oracle_geom* g) {
  if (!a || !g) return OR_NULL;
  memset(g, 0, sizeof(*g));
  if (a->rank < 3 || a->rank > 5) return OR_BAD_RANK;
  const int sr = a->rank - 2;
  g->spatial_rank = sr;
  if (a->n_strides && a->n_strides != sr) return OR_ATTR_LENGTH;
  if (a->n_dilations && a->n_dilations != sr) return OR_ATTR_LENGTH;
  if (a->n_pads && a->n_pads != 2 * sr) return OR_ATTR_LENGTH;
  if (a->n_output_padding && a->n_output_padding != sr) return OR_ATTR_LENGTH;
  for (int j = 0; j < 3; ++j) {
    const int ax = j - (3 - sr);
    int64_t op = 0;
    if (ax < 0) {
      g->in[j] = 1; g->k[j] = 1; g->s[j] = 1; g->d[j] = 1;
    } else {
      g->in[j] = a->x_shape[2 + ax];
      g->k[j] = a->w_shape[2 + ax];
      g->s[j] = a->n_strides ? a->strides[ax] : 1;
      g->d[j] = a->n_dilations ? a->dilations[ax] : 1;
      g->pad_begin[j] = a->n_pads ? a->pads[ax] : 0;
      g->pad_end[j] = a->n_pads ? a->pads[sr + ax] : 0;
      op = a->n_output_padding ? a->output_padding[ax] : 0;
    }
    if (g->k[j] < 1 || g->s[j] < 1 || g->d[j] < 1) return OR_ATTR_VALUE;
    if (g->pad_begin[j] < 0 || g->pad_end[j] < 0) return OR_ATTR_VALUE;
    if (op < 0 || op >= g->s[j]) return OR_ATTR_VALUE;
    g->out[j] = (g->in[j] - 1) * g->s[j] - g->pad_begin[j] - g->pad_end[j] +
                g->d[j] * (g->k[j] - 1) + op + 1;
  }
  /* every attribute value is checked before any output extent, as for the direct form */
  for (int j = 0; j < 3; ++j)
    if (g->out[j] < 1) return OR_EMPTY_OUTPUT;
  g->N = a->x_shape[0];
  g->C = a->x_shape[1];
  g->G = a->group;
  if (g->G < 1 || a->w_shape[0] != g->C || g->C % g->G != 0) return OR_GROUP;
  g->Cg = g->C / g->G;
  g->Mg = a->w_shape[1];
  g->M = g->Mg * g->G;
  if (g->N < 1 || g->C < 1 || g->Mg < 1) return OR_BAD_RANK;
  /* the activation and its parameters, as for the direct convolution */
  oracle_attrs t;
  memset(&t, 0, sizeof(t));
  t.activation = a->activation;
  t.n_act_params = a->n_act_params;
  t.act_params[0] = a->act_params[0];
  t.act_params[1] = a->act_params[1];
  const int act = t.activation, np = t.n_act_params;
  if (act < 0 || act >= A_COUNT) return OR_ACTIVATION;
  if (act == A_LEAKYRELU && np != 1) return OR_ACT_PARAMS;
  if ((act == A_HARDSIGMOID || act == A_CLIP) && np != 2) return OR_ACT_PARAMS;
  if ((act == A_QUICKGELU || act == A_ELU || act == A_THRESHOLDEDRELU || act == A_GELU) && np > 1)
    return OR_ACT_PARAMS;
  double alpha = 0.0, beta = 0.0;
  if (act == A_HARDSIGMOID) { alpha = 0.2; beta = 0.5; }
  else if (act == A_LEAKYRELU) alpha = 0.01;
  else if (act == A_QUICKGELU) alpha = 1.702;
  else if (act == A_ELU || act == A_THRESHOLDEDRELU) alpha = 1.0;
  if (np >= 1) alpha = t.act_params[0];
  if (np >= 2) beta = t.act_params[1];
  g->alpha = alpha;
  g->beta = beta;
  return OR_OK;
}

int oracle_transpose_output_shape(const oracle_tattrs* a, int64_t* y_shape) {
  oracle_geom g;
  const int st = oracle_resolve_transpose(a, &g);
  if (st != OR_OK) return st;
  y_shape[0] = g.N;
  y_shape[1] = g.M;
  for (int i = 0; i < g.spatial_rank; ++i) y_shape[2 + i] = g.out[3 - g.spatial_rank + i];
  return OR_OK;
}

/*
 * Scatter form: for every n, input channel c (group grp = c / Cg), output channel
 * m = grp*Mg + mm, input position i and tap t,
 *   s[n, m, i*stride - pad_begin + t*dilation] += x[n, c, i] * w[c, mm, t]
 * when that output position exists; then y = act(s + b[m] + z). abssum accumulates
 * |x * w| over the same terms. (n, group) pairs write disjoint outputs, so they run in
 * parallel.
 */
int oracle_conv_transpose(const oracle_tattrs* a, const double* x, const double* w,
                          const double* b, const double* z, double* y, double* abssum,
                          int nthreads) {
  oracle_geom g;
  const int st = oracle_resolve_transpose(a, &g);
  if (st != OR_OK) return st;
  if (!x || !w || !y) return OR_NULL;
  const int64_t ID = g.in[0], IH = g.in[1], IW = g.in[2];
  const int64_t KD = g.k[0], KH = g.k[1], KW = g.k[2];
  const int64_t OD = g.out[0], OH = g.out[1], OW = g.out[2];
  const int64_t P = OD * OH * OW, IS = ID * IH * IW, KS = KD * KH * KW;
  double* acc = (double*)calloc((size_t)(g.N * g.M * P), sizeof(double));
  double* aacc = (double*)calloc((size_t)(g.N * g.M * P), sizeof(double));
  if (!acc || !aacc) {
    free(acc);
    free(aacc);
    return OR_NULL;
  }
  const int64_t NG = g.N * g.G;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int64_t ng = 0; ng < NG; ++ng) {
    const int64_t n = ng / g.G, grp = ng % g.G;
    for (int64_t cc = 0; cc < g.Cg; ++cc) {
      const int64_t c = grp * g.Cg + cc;
      const double* xp = x + (n * g.C + c) * IS;
      for (int64_t mm = 0; mm < g.Mg; ++mm) {
        const int64_t m = grp * g.Mg + mm;
        const double* wp = w + (c * g.Mg + mm) * KS;
        double* sp = acc + (n * g.M + m) * P;
        double* ap = aacc + (n * g.M + m) * P;
        for (int64_t iz = 0; iz < ID; ++iz)
          for (int64_t iy = 0; iy < IH; ++iy)
            for (int64_t ix = 0; ix < IW; ++ix) {
              const double xv = xp[(iz * IH + iy) * IW + ix];
              for (int64_t kz = 0; kz < KD; ++kz) {
                const int64_t oz = iz * g.s[0] - g.pad_begin[0] + kz * g.d[0];
                if (oz < 0 || oz >= OD) continue;
                for (int64_t ky = 0; ky < KH; ++ky) {
                  const int64_t oy = iy * g.s[1] - g.pad_begin[1] + ky * g.d[1];
                  if (oy < 0 || oy >= OH) continue;
                  for (int64_t kx = 0; kx < KW; ++kx) {
                    const int64_t ox = ix * g.s[2] - g.pad_begin[2] + kx * g.d[2];
                    if (ox < 0 || ox >= OW) continue;
                    const double p = xv * wp[(kz * KH + ky) * KW + kx];
                    const int64_t o = (oz * OH + oy) * OW + ox;
                    sp[o] += p;
                    ap[o] += fabs(p);
                  }
                }
              }
            }
      }
    }
  }
  for (int64_t i = 0; i < g.N * g.M * P; ++i) {
    const int64_t m = (i / P) % g.M;
    double v = acc[i];
    if (b) v += b[m];
    if (z) v += z[i];
    y[i] = oracle_activation(a->activation, v, g.alpha, g.beta);
    if (abssum) abssum[i] = aacc[i];
  }
  free(acc);
  free(aacc);
  return OR_OK;
}

/* Number of OpenMP threads a parallel region would use (1 without OpenMP). */
int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
