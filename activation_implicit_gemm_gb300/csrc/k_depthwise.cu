// Depthwise 2-D FusedConv (C == M == group, one input and one output channel per group)
// on CUDA cores, bandwidth-first: the package's grouped large-kernel route
// (conv2d-grouped-large-w4: a shared input window held in registers, a 4-wide output
// vector per thread, bias seeding the accumulators, f32 accumulation) restated for
// GB300.
//
// One CTA per (image, channel, band of output rows). The CTA stages the band's input
// rows, zero-padded left/right/top/bottom, in shared memory as fp32; each thread then
// produces runs of VW consecutive outputs of one row from a register window of
// VW + KW - 1 input values per kernel row; bias, residual Z, the activation and the
// cast to T are applied before the store.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "epilogue.cuh"
#include "fconv_internal.h"

namespace fconv {

namespace {

constexpr int kDwThreads = 256;
constexpr int kDwMaxSmem = 96 * 1024;

struct DwLaunch {
  int band;      // output rows per CTA
  int bands;     // CTAs per (n, c) plane
  int srows;     // staged input rows
  int scols;     // staged input columns (padded width)
  size_t smem;
};

DwLaunch dw_shape(const ConvGeom& g) {
  DwLaunch L;
  L.scols = (g.OW - 1) * g.sW + (g.KW - 1) * g.dW + 1;
  L.band = g.OH;
  for (;;) {
    L.srows = (L.band - 1) * g.sH + (g.KH - 1) * g.dH + 1;
    L.smem = (size_t)L.srows * L.scols * sizeof(float) + (size_t)g.KH * g.KW * sizeof(float);
    if (L.smem <= (size_t)kDwMaxSmem || L.band == 1) break;
    L.band = (L.band + 1) / 2;
  }
  L.bands = (g.OH + L.band - 1) / L.band;
  return L;
}

template <typename T>
__device__ __forceinline__ void stage_input(const ConvGeom& g, const T* __restrict__ xp,
                                            float* sx, int row0, int srows, int scols) {
  const int total = srows * scols;
  for (int i = threadIdx.x; i < total; i += blockDim.x) {
    const int r = i / scols, c = i - r * scols;
    const int iy = row0 + r, ix = c - g.pW;
    float v = 0.0f;
    if (iy >= 0 && iy < g.IH && ix >= 0 && ix < g.IW) v = to_f32(xp[(long long)iy * g.IW + ix]);
    sx[i] = v;
  }
}

// + Z, activation and rounding of one run of up to VW outputs (activation fixed at
// compile time; f16 outputs use the fast exponentials).
template <int ACT, typename T, int VW>
__device__ __forceinline__ void store_run(const float (&acc)[VW], const T* __restrict__ z,
                                          T* __restrict__ y, long long o, int nv, float alpha,
                                          float beta) {
  float zv[VW];
#pragma unroll
  for (int j = 0; j < VW; ++j) zv[j] = (z && j < nv) ? to_f32(z[o + j]) : 0.0f;
#pragma unroll
  for (int j = 0; j < VW; ++j)
    if (j < nv)
      y[o + j] = from_f32<T>(act_eval<ACT, sizeof(T) == 2>(acc[j] + zv[j], alpha, beta));
}

// Fast path: stride 1 and dilation 1 along W, KW known at compile time.
template <typename T, int KW, int VW>
__global__ void __launch_bounds__(kDwThreads) dw_kernel_fast(ConvGeom g, const T* __restrict__ x,
                                                             const T* __restrict__ w,
                                                             const T* __restrict__ b,
                                                             const T* __restrict__ z,
                                                             T* __restrict__ y, int band,
                                                             int bands, int srows, int scols) {
  extern __shared__ float smem[];
  float* sw = smem;                       // KH*KW weights
  float* sx = smem + g.KH * KW;           // staged input
  const int plane = blockIdx.x / bands;   // n*C + c
  const int bi = blockIdx.x - plane * bands;
  const int c = plane % g.C;
  const int oh0 = bi * band;
  const int nrows = min(band, g.OH - oh0);
  const int row0 = oh0 * g.sH - g.pH;
  const T* xp = x + (long long)plane * g.IS;
  for (int i = threadIdx.x; i < g.KH * KW; i += blockDim.x) sw[i] = to_f32(w[(long long)c * g.KH * KW + i]);
  stage_input(g, xp, sx, row0, srows, scols);
  __syncthreads();
  const float bias = b ? to_f32(b[c]) : 0.0f;
  const int runs_per_row = (g.OW + VW - 1) / VW;
  const int runs = nrows * runs_per_row;
  const long long ybase = (long long)plane * g.P;
  for (int r = threadIdx.x; r < runs; r += blockDim.x) {
    const int orow = r / runs_per_row;
    const int ow0 = (r - orow * runs_per_row) * VW;
    const int oh = oh0 + orow;
    float acc[VW];
#pragma unroll
    for (int j = 0; j < VW; ++j) acc[j] = bias;
    const float* srow = sx + (orow * g.sH) * scols + ow0;
    for (int ky = 0; ky < g.KH; ++ky) {
      const float* s = srow + ky * g.dH * scols;
      float win[VW + KW - 1];
#pragma unroll
      for (int i = 0; i < VW + KW - 1; ++i) win[i] = (ow0 + i < scols) ? s[i] : 0.0f;
      const float* wr = sw + ky * KW;
#pragma unroll
      for (int kx = 0; kx < KW; ++kx) {
        const float wv = wr[kx];
#pragma unroll
        for (int j = 0; j < VW; ++j) acc[j] = fmaf(win[j + kx], wv, acc[j]);
      }
    }
    const long long o = ybase + (long long)oh * g.OW + ow0;
    const int nv = min(VW, g.OW - ow0);
#define FCONV_DW_STORE(ACT) store_run<ACT, T, VW>(acc, z, y, o, nv, g.alpha, g.beta)
    FCONV_ACT_SWITCH(g.act, FCONV_DW_STORE)
#undef FCONV_DW_STORE
  }
}

// General path: any stride and dilation, one output per thread iteration.
template <typename T>
__global__ void __launch_bounds__(kDwThreads) dw_kernel_generic(ConvGeom g, const T* __restrict__ x,
                                                                const T* __restrict__ w,
                                                                const T* __restrict__ b,
                                                                const T* __restrict__ z,
                                                                T* __restrict__ y, int band,
                                                                int bands, int srows, int scols) {
  extern __shared__ float smem[];
  float* sw = smem;
  float* sx = smem + g.KH * g.KW;
  const int plane = blockIdx.x / bands;
  const int bi = blockIdx.x - plane * bands;
  const int c = plane % g.C;
  const int oh0 = bi * band;
  const int nrows = min(band, g.OH - oh0);
  const int row0 = oh0 * g.sH - g.pH;
  const T* xp = x + (long long)plane * g.IS;
  for (int i = threadIdx.x; i < g.KH * g.KW; i += blockDim.x)
    sw[i] = to_f32(w[(long long)c * g.KH * g.KW + i]);
  stage_input(g, xp, sx, row0, srows, scols);
  __syncthreads();
  const float bias = b ? to_f32(b[c]) : 0.0f;
  const int outs = nrows * g.OW;
  const long long ybase = (long long)plane * g.P;
  for (int i = threadIdx.x; i < outs; i += blockDim.x) {
    const int orow = i / g.OW, ow = i - orow * g.OW;
    float acc = bias;
    for (int ky = 0; ky < g.KH; ++ky) {
      const float* s = sx + (orow * g.sH + ky * g.dH) * scols + ow * g.sW;
      for (int kx = 0; kx < g.KW; ++kx) acc = fmaf(s[kx * g.dW], sw[ky * g.KW + kx], acc);
    }
    const long long o = ybase + (long long)(oh0 + orow) * g.OW + ow;
    float v = acc;
    if (z) v += to_f32(z[o]);
    y[o] = from_f32<T>(apply_act(g.act, v, g.alpha, g.beta));
  }
}

template <typename T>
int launch_dw_t(const ConvGeom& g, const ConvArgs& a, cudaStream_t s) {
  const DwLaunch L = dw_shape(g);
  const long long blocks = (long long)g.N * g.C * L.bands;
  const T* x = (const T*)a.x;
  const T* w = (const T*)a.w;
  const T* b = (const T*)a.b;
  const T* z = (const T*)a.z;
  T* y = (T*)a.y;
  const bool unit = g.sW == 1 && g.dW == 1;
#define FCONV_DW_FAST(KWV)                                                                   \
  if (unit && g.KW == KWV) {                                                                 \
    auto k = dw_kernel_fast<T, KWV, 4>;                                                      \
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.smem);      \
    k<<<(unsigned)blocks, kDwThreads, L.smem, s>>>(g, x, w, b, z, y, L.band, L.bands, L.srows, \
                                                    L.scols);                                \
    return (int)cudaGetLastError();                                                          \
  }
  FCONV_DW_FAST(3)
  FCONV_DW_FAST(5)
  FCONV_DW_FAST(7)
#undef FCONV_DW_FAST
  auto k = dw_kernel_generic<T>;
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.smem);
  k<<<(unsigned)blocks, kDwThreads, L.smem, s>>>(g, x, w, b, z, y, L.band, L.bands, L.srows,
                                                  L.scols);
  return (int)cudaGetLastError();
}

}  // namespace

bool depthwise_supported(const ConvGeom& g) {
  if (!(g.Cg == 1 && g.Mg == 1 && g.KD == 1 && g.ID == 1 && g.OD == 1)) return false;
  const long long blocks = (long long)g.N * g.C * dw_shape(g).bands;
  if (blocks > 0x7fffffffLL) return false;
  return dw_shape(g).smem <= (size_t)kDwMaxSmem;
}

int launch_depthwise(const ConvGeom& g, const ConvArgs& a, void* stream) {
  cudaStream_t s = (cudaStream_t)stream;
  if (g.dtype == FCONV_F16) return launch_dw_t<__half>(g, a, s);
  return launch_dw_t<float>(g, a, s);
}

}  // namespace fconv
