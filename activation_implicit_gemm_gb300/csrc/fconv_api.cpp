// FusedConv planner and C ABI (include/fconv.h).
//
// fconv_plan_create validates a request with the rules of the com.microsoft.FusedConv
// manifest (derive: kernelShapeLengthOk .. padsLengthOk, kernelShapeMatchesWeights,
// kernelExtentsOk, stridesValuesOk, dilationsValuesOk, padsValuesOk, explicitPadsOk,
// groupOk, biasOk, zOk, activationOk, activationParamsOk), resolves the applied pads and
// output sizes (samePad*, samePadFront/Top/Left, effectivePad*, expectedOutput*) and
// picks a kernel route. Nothing is allocated on the device and nothing is launched
// until fconv_run.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>

#include "fastdiv.cuh"
#include "fconv_internal.h"

using namespace fconv;

struct fconv_plan {
  fconv_desc desc;
  ConvGeom g;
  int rank;
  int64_t y_shape[5];
  int64_t pad_begin[3], pad_end[3];
  fconv_route route;
  IgemmConfig igemm;
  size_t workspace;
  int sms;
  double flops;   // algorithmic FLOPs of one run
};

namespace {

int64_t floordiv(int64_t a, int64_t b) {
  int64_t q = a / b;
  if ((a % b != 0) && (a < 0)) q -= 1;
  return q;
}

int device_sms(int device) {
  int count = 0;
  if (cudaGetDeviceCount(&count) != cudaSuccess || count <= 0) {
    cudaGetLastError();
    return 152;
  }
  int dev = device;
  if (dev < 0 && cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 152;
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      sms <= 0) {
    cudaGetLastError();
    return 152;
  }
  return sms;
}

bool fits_int(int64_t v) { return v >= 0 && v <= INT_MAX; }

// Attribute and shape rules, in the order the status codes are documented.
fconv_status resolve(const fconv_desc* d, fconv_plan* p) {
  if (d->dtype != FCONV_F32 && d->dtype != FCONV_F16) return FCONV_E_UNSUPPORTED;
  if (d->rank < 3 || d->rank > 5) return FCONV_E_RANK;
  const int r = d->rank, sr = r - 2;
  for (int i = 0; i < r; ++i)
    if (d->x_shape[i] < 1 || d->w_shape[i] < 1) return FCONV_E_RANK;
  if ((d->n_kernel_shape && d->n_kernel_shape != sr) || (d->n_strides && d->n_strides != sr) ||
      (d->n_dilations && d->n_dilations != sr) || (d->n_pads && d->n_pads != 2 * sr) ||
      (d->n_output_padding && d->n_output_padding != sr))
    return FCONV_E_ATTR_LENGTH;
  const bool tr = d->transposed != 0;
  int64_t in[3], k[3], s[3], dl[3], pb[3], pe[3], out[3], op[3];
  for (int j = 0; j < 3; ++j) {
    const int ax = j - (3 - sr);
    if (ax < 0) {
      in[j] = k[j] = s[j] = dl[j] = 1;
      pb[j] = pe[j] = op[j] = 0;
      continue;
    }
    op[j] = d->n_output_padding ? d->output_padding[ax] : 0;
    in[j] = d->x_shape[2 + ax];
    k[j] = d->w_shape[2 + ax];
    s[j] = d->n_strides ? d->strides[ax] : 1;
    dl[j] = d->n_dilations ? d->dilations[ax] : 1;
    pb[j] = d->n_pads ? d->pads[ax] : 0;
    pe[j] = d->n_pads ? d->pads[sr + ax] : 0;
    if (d->n_kernel_shape && d->kernel_shape[ax] != k[j]) return FCONV_E_KERNEL_SHAPE;
  }
  for (int j = 0; j < 3; ++j)
    if (s[j] < 1 || dl[j] < 1 || pb[j] < 0 || pe[j] < 0 || k[j] < 1) return FCONV_E_ATTR_VALUE;
  if (d->auto_pad < FCONV_PAD_NOTSET || d->auto_pad > FCONV_PAD_VALID) return FCONV_E_ATTR_VALUE;
  if (d->auto_pad != FCONV_PAD_NOTSET && d->n_pads) return FCONV_E_PADS_WITH_AUTOPAD;
  // output_padding: below the stride on the transposed form, zero on the direct one
  for (int j = 0; j < 3; ++j)
    if (op[j] < 0 || (tr ? op[j] >= s[j] : op[j] != 0)) return FCONV_E_ATTR_VALUE;
  if (tr && (d->auto_pad == FCONV_PAD_SAME_UPPER || d->auto_pad == FCONV_PAD_SAME_LOWER))
    return FCONV_E_UNSUPPORTED;
  for (int j = 0; j < 3 && tr; ++j) {
    if (d->auto_pad == FCONV_PAD_VALID) pb[j] = pe[j] = 0;
    out[j] = (in[j] - 1) * s[j] - pb[j] - pe[j] + dl[j] * (k[j] - 1) + op[j] + 1;
    if (out[j] < 1) return FCONV_E_OUTPUT_EMPTY;
  }
  for (int j = 0; j < 3 && !tr; ++j) {
    const int64_t ext = (k[j] - 1) * dl[j] + 1;
    if (d->auto_pad == FCONV_PAD_SAME_UPPER || d->auto_pad == FCONV_PAD_SAME_LOWER) {
      out[j] = (in[j] + s[j] - 1) / s[j];
      int64_t total = (out[j] - 1) * s[j] + ext - in[j];
      if (total < 0) total = 0;
      const int64_t lo = total / 2;
      pb[j] = d->auto_pad == FCONV_PAD_SAME_UPPER ? lo : total - lo;
      pe[j] = total - pb[j];
    } else {
      if (d->auto_pad == FCONV_PAD_VALID) pb[j] = pe[j] = 0;
      out[j] = floordiv(in[j] + pb[j] + pe[j] - ext, s[j]) + 1;
    }
    if (out[j] < 1) return FCONV_E_OUTPUT_EMPTY;
  }
  const int64_t N = d->x_shape[0], C = d->x_shape[1], G = d->group;
  const int64_t M = tr ? d->w_shape[1] * G : d->w_shape[0];
  if (tr) {
    if (G < 1 || d->w_shape[0] != C || C % G != 0) return FCONV_E_GROUP;
  } else if (G < 1 || M % G != 0 || d->w_shape[1] * G != C) {
    return FCONV_E_GROUP;
  }
  if (d->has_bias && d->bias_len != M) return FCONV_E_BIAS_SHAPE;

  const int act = (int)d->activation, np = d->n_act_params;
  if (act < FCONV_ACT_NONE || act > FCONV_ACT_ERF) return FCONV_E_ACTIVATION;
  if (np > 2) return FCONV_E_ACT_PARAMS;
  if (act == FCONV_ACT_LEAKYRELU && np != 1) return FCONV_E_ACT_PARAMS;
  if ((act == FCONV_ACT_HARDSIGMOID || act == FCONV_ACT_CLIP) && np != 2) return FCONV_E_ACT_PARAMS;
  if ((act == FCONV_ACT_QUICKGELU || act == FCONV_ACT_ELU || act == FCONV_ACT_THRESHOLDEDRELU ||
       act == FCONV_ACT_GELU) && np > 1)
    return FCONV_E_ACT_PARAMS;
  float alpha = 0.0f, beta = 0.0f;  // defaults: manifest derive actAlpha / actBeta
  if (act == FCONV_ACT_HARDSIGMOID) { alpha = 0.2f; beta = 0.5f; }
  else if (act == FCONV_ACT_LEAKYRELU) alpha = 0.01f;
  else if (act == FCONV_ACT_QUICKGELU) alpha = 1.702f;
  else if (act == FCONV_ACT_ELU || act == FCONV_ACT_THRESHOLDEDRELU) alpha = 1.0f;
  if (np >= 1) alpha = d->act_params[0];
  if (np >= 2) beta = d->act_params[1];

  p->rank = r;
  p->y_shape[0] = N;
  p->y_shape[1] = M;
  for (int i = 0; i < sr; ++i) p->y_shape[2 + i] = out[3 - sr + i];
  for (int j = 0; j < 3; ++j) { p->pad_begin[j] = pb[j]; p->pad_end[j] = pe[j]; }
  if (d->has_z) {
    if (d->z_rank != r) return FCONV_E_Z_SHAPE;
    for (int i = 0; i < r; ++i)
      if (d->z_shape[i] != p->y_shape[i]) return FCONV_E_Z_SHAPE;
  }

  // Geometry in 32-bit ints (tensor-level offsets stay 64-bit in the kernels).
  const int64_t vals[] = {N, C, M, G, in[0], in[1], in[2], out[0], out[1], out[2], k[0], k[1],
                          k[2], s[0], s[1], s[2], dl[0], dl[1], dl[2], pb[0], pb[1], pb[2]};
  for (int64_t v : vals)
    if (!fits_int(v)) return FCONV_E_UNSUPPORTED;
  const int64_t KV = k[0] * k[1] * k[2];
  const int64_t Kg = (C / G) * KV;
  if (!fits_int(KV) || !fits_int(Kg)) return FCONV_E_UNSUPPORTED;
  ConvGeom& g = p->g;
  g.dtype = d->dtype;
  g.N = (int)N; g.C = (int)C; g.M = (int)M; g.G = (int)G;
  g.Cg = (int)(C / G); g.Mg = (int)(M / G);
  g.ID = (int)in[0]; g.IH = (int)in[1]; g.IW = (int)in[2];
  g.OD = (int)out[0]; g.OH = (int)out[1]; g.OW = (int)out[2];
  g.KD = (int)k[0]; g.KH = (int)k[1]; g.KW = (int)k[2];
  g.sD = (int)s[0]; g.sH = (int)s[1]; g.sW = (int)s[2];
  g.dD = (int)dl[0]; g.dH = (int)dl[1]; g.dW = (int)dl[2];
  g.pD = (int)pb[0]; g.pH = (int)pb[1]; g.pW = (int)pb[2];
  g.act = act; g.alpha = alpha; g.beta = beta;
  g.transposed = tr ? 1 : 0;
  // FLOPs: 2 * N * M * P * Kg for the direct form (every tap of every output); for the
  // transposed form 2 * N * C * M/group * the (input position, tap) pairs that land on an
  // output, counted per axis
  if (tr) {
    double pairs = 1.0;
    for (int j = 0; j < 3; ++j) {
      int64_t cnt = 0;
      for (int64_t i = 0; i < in[j]; ++i)
        for (int64_t t = 0; t < k[j]; ++t) {
          const int64_t o = i * s[j] - pb[j] + t * dl[j];
          if (o >= 0 && o < out[j]) ++cnt;
        }
      pairs *= (double)cnt;
    }
    p->flops = 2.0 * (double)N * (double)C * (double)(M / G) * pairs;
  } else {
    p->flops = 2.0 * (double)N * (double)M * (double)(out[0] * out[1] * out[2]) * (double)Kg;
  }
  g.has_bias = d->has_bias ? 1 : 0;
  g.has_z = d->has_z ? 1 : 0;
  g.P = (long long)(out[0] * out[1] * out[2]);
  g.IS = (long long)(in[0] * in[1] * in[2]);
  g.KV = (int)KV;
  g.Kg = (int)Kg;
  return FCONV_OK;
}

// Largest pixel tile (MMA N) of the tensor-core kernels; channel tiles are always 128.
constexpr int kDefaultPixelTile = 256;
// FLOPs per HBM byte above which a GB300 conv is tensor-bound: the measured dense f16 GEMM
// rate over the measured copy rate (1909 TFLOP/s / 6787 GB/s).
constexpr double kRidgeFlopPerByte = 281.0;

void plan_igemm(fconv_plan* p, const fconv_options* o) {
  const ConvGeom& g = p->g;
  IgemmConfig& c = p->igemm;
  c.tile_n = (o && o->tile_n) ? o->tile_n : kDefaultPixelTile;
  c.a_path = igemm_tc_resolve_path(g, c.tile_n, o ? o->a_path : 0);
  if (!(o && o->tile_n) && c.a_path == 2 && g.dtype == FCONV_F16) {
    // TMA-fed convs below the ridge (HBM-bound) run faster with more, smaller pixel tiles:
    // measured on the suite, 256 -> 128 pixels took cnn B (64->128 @16) from 46 to 41 us and
    // the stem downsample from 28 to 25 us, and 64 pixels took the 1-D conv (16 tiles of
    // 256) from 24 to 13 us; the tensor-bound convs keep 256
    const double flops = 2.0 * g.N * (double)g.M * (double)g.P * g.Kg;
    const double bytes = 2.0 * ((double)g.N * g.C * (double)g.IS + (double)g.M * g.Kg +
                                (double)g.N * g.M * (double)g.P * (g.has_z ? 2.0 : 1.0));
    if (flops < kRidgeFlopPerByte * bytes) {
      c.tile_n = 128;
      const long long units = igemm_tc_mtiles(g, 2, 128) * ((g.Mg + 127) / 128) * g.G;
      if (units * 2 < p->sms) c.tile_n = 64;
    }
  }
  const long long rows = igemm_tc_mtiles(g, c.a_path, c.tile_n);
  const long long tiles = rows * ((g.Mg + 127) / 128) * g.G;
  const int chunks = igemm_tc_chunks(g, c.a_path, c.tile_n);
  int split = 1;
  if (o && o->split_k > 0) {
    split = o->split_k;
  } else if (tiles * 2 <= p->sms && chunks >= 8) {
    // one persistent CTA per SM: split K only when at least two splits fit per tile and K
    // is long enough (8+ chunks) for the partials' round trip and the reduce launch to pay
    long long s = p->sms / tiles;
    if (s > chunks) s = chunks;
    if (s > 16) s = 16;
    split = (int)(s < 1 ? 1 : s);
  }
  if (split > chunks) split = chunks;
  if (split < 1) split = 1;
  // no empty split: every split gets ceil(chunks / split) chunks except possibly the last
  const int per = (chunks + split - 1) / split;
  split = (chunks + per - 1) / per;
  c.split_k = split;
  const long long units = tiles * split;
  c.grid = units < p->sms ? units : p->sms;
  if (g.max_ctas > 0 && c.grid > g.max_ctas) c.grid = g.max_ctas;
  p->workspace = igemm_tc_workspace_bytes(g, c);
}

fconv_status create(const fconv_desc* d, int device, const fconv_options* o, fconv_plan** out) {
  if (!out) return FCONV_E_NULL;
  *out = nullptr;
  if (!d) return FCONV_E_NULL;
  fconv_plan* p = new (std::nothrow) fconv_plan();
  if (!p) return FCONV_E_NOMEM;
  std::memset(p, 0, sizeof(*p));
  p->desc = *d;
  fconv_status st = resolve(d, p);
  if (st != FCONV_OK) {
    delete p;
    return st;
  }
  p->sms = device_sms(device);
  if (o && o->max_ctas < 0) {
    delete p;
    return FCONV_E_UNSUPPORTED;
  }
  p->g.max_ctas = o ? o->max_ctas : 0;
  p->g.precision = o ? o->precision : FCONV_PRECISION_DEFAULT;
  if (p->g.precision != FCONV_PRECISION_DEFAULT &&
      (p->g.precision != FCONV_PRECISION_HALF2_ROWS || !depthwise_half2_supported(p->g))) {
    delete p;
    return FCONV_E_UNSUPPORTED;
  }
  const fconv_route want = o ? o->route : FCONV_ROUTE_AUTO;
  fconv_route route = want;
  const int tile_n = (o && o->tile_n) ? o->tile_n : kDefaultPixelTile;
  // groups with few channels and short reductions (C/group * kernel <= 64, e.g. 1-D and 3-D
  // depthwise) do few FMAs per output: CUDA cores with a shared-memory halo box (2-D
  // depthwise has a kernel of its own). Longer group reductions go to the tensor cores,
  // which were faster on the 3-D grouped conv X[2,32,16,64,64] W[64,8,3,3,3] group 4
  // (C/group * kernel = 216).
  const bool small_groups = p->g.G > 1 && p->g.Cg <= 16 && p->g.Mg <= 32 && p->g.Kg <= 64;
  if (p->g.transposed) {
    // the transposed form has one route
    if ((want != FCONV_ROUTE_AUTO && want != FCONV_ROUTE_TRANSPOSED) ||
        !transposed_supported(p->g))
      st = FCONV_E_UNSUPPORTED;
    route = FCONV_ROUTE_TRANSPOSED;
  } else if (want == FCONV_ROUTE_AUTO) {
    if (depthwise_supported(p->g)) route = FCONV_ROUTE_DEPTHWISE;
    else if (small_groups && grouped_supported(p->g)) route = FCONV_ROUTE_GROUPED;
    else if (igemm_tc_supported(p->g, tile_n)) route = FCONV_ROUTE_IGEMM_TC;
    else route = FCONV_ROUTE_DIRECT;
  } else if (want == FCONV_ROUTE_DEPTHWISE && !depthwise_supported(p->g)) {
    st = FCONV_E_UNSUPPORTED;
  } else if (want == FCONV_ROUTE_GROUPED && !grouped_supported(p->g)) {
    st = FCONV_E_UNSUPPORTED;
  } else if (want == FCONV_ROUTE_IGEMM_TC && !igemm_tc_supported(p->g, tile_n)) {
    st = FCONV_E_UNSUPPORTED;
  } else if (want != FCONV_ROUTE_DIRECT && want != FCONV_ROUTE_DEPTHWISE &&
             want != FCONV_ROUTE_IGEMM_TC && want != FCONV_ROUTE_GROUPED) {
    // includes FCONV_ROUTE_TRANSPOSED for a direct convolution
    st = FCONV_E_UNSUPPORTED;
  }
  // the half2 mode exists on the depthwise kernel only
  if (st == FCONV_OK && p->g.precision != FCONV_PRECISION_DEFAULT && route != FCONV_ROUTE_DEPTHWISE)
    st = FCONV_E_UNSUPPORTED;
  if (st == FCONV_OK && route == FCONV_ROUTE_IGEMM_TC && o && o->tile_n &&
      o->tile_n != 64 && o->tile_n != 128 && o->tile_n != 256)
    st = FCONV_E_UNSUPPORTED;
  if (st == FCONV_OK && route == FCONV_ROUTE_IGEMM_TC && o &&
      (o->a_path < 0 || o->a_path > 2 || igemm_tc_resolve_path(p->g, tile_n, o->a_path) == 0))
    st = FCONV_E_UNSUPPORTED;
  if (st != FCONV_OK) {
    delete p;
    return st;
  }
  p->route = route;
  if (route == FCONV_ROUTE_IGEMM_TC) plan_igemm(p, o);
  if (std::getenv("FCONV_LOG")) {
    std::fprintf(stderr, "[fconv] route=%d tile_n=%d split_k=%d ws=%zu sms=%d Kg=%d Mg=%d\n",
                 (int)route, p->igemm.tile_n, p->igemm.split_k, p->workspace, p->sms, p->g.Kg,
                 p->g.Mg);
  }
  *out = p;
  return FCONV_OK;
}

bool misaligned(const void* ptr) { return ((uintptr_t)ptr & 15u) != 0; }

}  // namespace

extern "C" {

fconv_status fconv_plan_create(const fconv_desc* desc, int device, fconv_plan** out) {
  return create(desc, device, nullptr, out);
}

fconv_status fconv_plan_create_ex(const fconv_desc* desc, int device, const fconv_options* opts,
                                  fconv_plan** out) {
  return create(desc, device, opts, out);
}

fconv_status fconv_plan_output_shape(const fconv_plan* p, int64_t y_shape[5], int* rank) {
  if (!p || !y_shape || !rank) return FCONV_E_NULL;
  for (int i = 0; i < 5; ++i) y_shape[i] = i < p->rank ? p->y_shape[i] : 0;
  *rank = p->rank;
  return FCONV_OK;
}

fconv_status fconv_plan_pads(const fconv_plan* p, int64_t pad_begin[3], int64_t pad_end[3]) {
  if (!p || !pad_begin || !pad_end) return FCONV_E_NULL;
  for (int j = 0; j < 3; ++j) {
    pad_begin[j] = p->pad_begin[j];
    pad_end[j] = p->pad_end[j];
  }
  return FCONV_OK;
}

fconv_status fconv_plan_workspace_size(const fconv_plan* p, size_t* bytes) {
  if (!p || !bytes) return FCONV_E_NULL;
  *bytes = p->workspace;
  return FCONV_OK;
}

fconv_status fconv_plan_route(const fconv_plan* p, fconv_route* route, int* tile_n,
                              int* split_k) {
  if (!p) return FCONV_E_NULL;
  if (route) *route = p->route;
  if (tile_n) *tile_n = p->route == FCONV_ROUTE_IGEMM_TC ? p->igemm.tile_n : 0;
  if (split_k) *split_k = p->route == FCONV_ROUTE_IGEMM_TC ? p->igemm.split_k : 1;
  return FCONV_OK;
}

fconv_status fconv_plan_launches(const fconv_plan* p, int* kernels) {
  if (!p || !kernels) return FCONV_E_NULL;
  *kernels = p->route == FCONV_ROUTE_IGEMM_TC ? igemm_tc_launches(p->g, p->igemm) : 1;
  return FCONV_OK;
}

fconv_status fconv_plan_work(const fconv_plan* p, double* flops, double* bytes) {
  if (!p) return FCONV_E_NULL;
  const ConvGeom& g = p->g;
  const double es = g.dtype == FCONV_F16 ? 2.0 : 4.0;
  const double ny = (double)g.N * g.M * (double)g.P;
  (void)ny;
  if (flops) *flops = p->flops;
  if (bytes) {
    double b = (double)g.N * g.C * (double)g.IS + (double)g.M * g.Kg + ny;
    if (g.has_bias) b += g.M;
    if (g.has_z) b += ny;
    *bytes = b * es;
  }
  return FCONV_OK;
}

fconv_status fconv_run(const fconv_plan* p, const void* x, const void* w, const void* b,
                       const void* z, void* y, void* workspace, size_t workspace_bytes,
                       void* stream) {
  if (!p || !x || !w || !y) return FCONV_E_NULL;
  if (p->g.has_bias && !b) return FCONV_E_NULL;
  if (!p->g.has_bias && b) return FCONV_E_BIAS_SHAPE;
  if (p->g.has_z && !z) return FCONV_E_NULL;
  if (!p->g.has_z && z) return FCONV_E_Z_SHAPE;
  if (misaligned(x) || misaligned(w) || misaligned(y) || (b && misaligned(b)) ||
      (z && misaligned(z)) || (workspace && misaligned(workspace)))
    return FCONV_E_ALIGNMENT;
  if (y == x || y == w || (b && y == b) || (z && y == z) || (workspace && y == workspace))
    return FCONV_E_ALIAS;
  if (p->workspace > 0 && (!workspace || workspace_bytes < p->workspace)) return FCONV_E_WORKSPACE;
  ConvArgs a{x, w, b, z, y, workspace};
  int err = 0;
  switch (p->route) {
    case FCONV_ROUTE_DIRECT: err = launch_direct(p->g, a, stream); break;
    case FCONV_ROUTE_DEPTHWISE: err = launch_depthwise(p->g, a, stream); break;
    case FCONV_ROUTE_GROUPED: err = launch_grouped(p->g, a, stream); break;
    case FCONV_ROUTE_TRANSPOSED: err = launch_transposed(p->g, a, stream); break;
    case FCONV_ROUTE_IGEMM_TC: err = launch_igemm_tc(p->g, p->igemm, a, stream); break;
    default: return FCONV_E_UNSUPPORTED;
  }
  return err == 0 ? FCONV_OK : FCONV_E_CUDA;
}

fconv_status fconv_check_device(void* stream) {
  unsigned v = 0;
  if (read_and_clear_device_error(stream, &v) != 0) return FCONV_E_CUDA;
  return v ? FCONV_E_DEVICE_TIMEOUT : FCONV_OK;
}

void fconv_destroy(fconv_plan* p) { delete p; }

const char* fconv_status_string(fconv_status s) {
  switch (s) {
    case FCONV_OK: return "ok";
    case FCONV_E_NULL: return "a required pointer is NULL";
    case FCONV_E_RANK: return "X and W must have the same rank 3..5 and positive extents";
    case FCONV_E_ATTR_LENGTH: return "an attribute has the wrong number of entries";
    case FCONV_E_ATTR_VALUE: return "strides/dilations must be >= 1, pads >= 0";
    case FCONV_E_PADS_WITH_AUTOPAD: return "pads cannot be combined with auto_pad";
    case FCONV_E_KERNEL_SHAPE: return "kernel_shape does not match W";
    case FCONV_E_GROUP: return "group must divide M and W.shape[1] * group must equal C";
    case FCONV_E_BIAS_SHAPE: return "bias must be rank 1 with length M";
    case FCONV_E_Z_SHAPE: return "Z must have the shape of Y";
    case FCONV_E_ACT_PARAMS: return "activation_params has the wrong number of values";
    case FCONV_E_ACTIVATION: return "unknown activation";
    case FCONV_E_OUTPUT_EMPTY: return "an output extent would be < 1";
    case FCONV_E_WORKSPACE: return "workspace too small";
    case FCONV_E_UNSUPPORTED: return "request not supported by this library or route";
    case FCONV_E_CUDA: return "CUDA error";
    case FCONV_E_DEVICE_TIMEOUT: return "a kernel gave up a bounded wait";
    case FCONV_E_NOMEM: return "out of host memory";
    case FCONV_E_ALIGNMENT: return "device pointers must be 16-byte aligned";
    case FCONV_E_ALIAS: return "Y must not alias an input or the workspace";
  }
  return "unknown status";
}

int fconv_version(void) { return 100; }

// Host-side check of the invariant-divisor arithmetic the kernels use (a test hook, not
// part of the documented ABI): 0 when every case agrees with ordinary division.
int fconv_selftest_fastdiv(void) {
  uint64_t state = 0x2545F4914F6CDD1Dull;
  for (uint32_t d = 1; d < 5000; ++d) {
    const FastDiv f = make_fastdiv(d);
    for (int t = 0; t < 400; ++t) {
      state ^= state << 13; state ^= state >> 7; state ^= state << 17;  // xorshift64
      uint32_t n = (uint32_t)(state & 0x7fffffffu);
      if (t < 8) n = (uint32_t)t * d + (uint32_t)(t & 1) * (d - 1);  // multiples and edges
      if (t == 8) n = 0x7fffffffu;
      if (fast_div(n, f) != n / d) return 1;
    }
  }
  const uint32_t big[] = {65535u, 65536u, 100352u, 524288u, 3136u, 784u, 1u << 20, 0x7fffffffu};
  for (uint32_t d : big) {
    const FastDiv f = make_fastdiv(d);
    for (uint32_t n : {0u, d - 1, d, 2 * d - 1, 0x7fffffffu, 0x7ffffffeu, 123456789u})
      if (fast_div(n, f) != n / d) return 2;
  }
  return 0;
}

}  // extern "C"
