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
#include "ptx.cuh"

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

// + Z, activation and rounding of a 4 x 4 block (rows nr, columns nv valid): all Z
// loads first, then the math, then the stores.
template <int ACT, typename T>
__device__ __forceinline__ void store_block4(const float (&acc)[4][4], const T* __restrict__ z,
                                             T* __restrict__ y, long long o, int OW, int nr,
                                             int nv, float alpha, float beta) {
  float zv[4][4];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int j = 0; j < 4; ++j)
      zv[r][j] = (z && r < nr && j < nv) ? to_f32(z[o + (long long)r * OW + j]) : 0.0f;
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (r < nr && j < nv)
        y[o + (long long)r * OW + j] =
            from_f32<T>(act_eval<ACT, sizeof(T) == 2>(acc[r][j] + zv[r][j], alpha, beta));
}

// Four consecutive outputs starting at p (p 4-element aligned): one 8-byte (f16) or
// 16-byte (f32) store.
__device__ __forceinline__ void store4(__half* p, const float (&v)[4]) {
  const __half2 a = __floats2half2_rn(v[0], v[1]), b = __floats2half2_rn(v[2], v[3]);
  uint2 r;
  r.x = *reinterpret_cast<const uint32_t*>(&a);
  r.y = *reinterpret_cast<const uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = r;
}
__device__ __forceinline__ void store4(float* p, const float (&v)[4]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}

// Activation, rounding and one vector store per row of a 4 x 4 block of whole runs.
template <int ACT, typename T>
__device__ __forceinline__ void store_rows4(const float (&acc)[4][4], T* __restrict__ y, long long o,
                                            int OW, int nr, float alpha, float beta) {
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    if (r < nr) {
      float v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = act_eval<ACT, sizeof(T) == 2>(acc[r][j], alpha, beta);
      store4(y + o + (long long)r * OW, v);
    }
  }
}

// Fast path: stride 1 and dilation 1 on both axes, KH and KW known at compile time.
// A CTA owns an output tile of TR x TC (both multiples of 4) of one (image, channel)
// plane; each thread computes a 4 x 4 block of outputs from KH + 3 input rows of
// KW + 3 values each, read as 16-byte vectors from the fp32 halo tile in shared memory
// (column c of the tile holds input column c - 4 + ox0 - pW, so every vector read of a
// thread starts 16-byte aligned). Weights live in registers; accumulation is fp32.
template <typename T, int KH, int KW>
__global__ void __launch_bounds__(256) dw_kernel_block(ConvGeom g, const T* __restrict__ x,
                                                       const T* __restrict__ w,
                                                       const T* __restrict__ b,
                                                       const T* __restrict__ z,
                                                       T* __restrict__ y, int TR, int TC,
                                                       int tiles_r, int tiles_c, int pitch) {
  ptx::pdl_wait();  // inputs may be the previous kernel's outputs
  ptx::pdl_trigger();
  extern __shared__ float sx[];  // (TR + KH - 1) rows x pitch floats
  constexpr int WIN = 4 + KW - 1;
  constexpr int WV = (WIN + 3 + 3) / 4;  // 16-byte vectors covering the window (+3 offset)
  const int tiles = tiles_r * tiles_c;
  const int plane = blockIdx.x / tiles;
  const int tile = blockIdx.x - plane * tiles;
  const int tr = tile / tiles_c, tc = tile - tr * tiles_c;
  const int oy0 = tr * TR, ox0 = tc * TC;
  const int c = plane % g.C;
  const T* xp = x + (long long)plane * g.IS;
  const int srows = TR + KH - 1;
  const int iy0 = oy0 - g.pH;          // input row of tile row 0
  const int ixb = ox0 - g.pW - 4;      // input column of tile column 0
  // zero the tile (padding), then copy the input rows it covers with 16-byte loads,
  // four in flight per thread
  for (int i = threadIdx.x * 4; i < srows * pitch; i += blockDim.x * 4)
    *reinterpret_cast<float4*>(sx + i) = make_float4(0.f, 0.f, 0.f, 0.f);
  float wr[KH * KW];
#pragma unroll
  for (int i = 0; i < KH * KW; ++i) wr[i] = to_f32(w[(long long)c * KH * KW + i]);
  const float bias = b ? to_f32(b[c]) : 0.0f;
  __syncthreads();
  {
    constexpr int VE = 16 / sizeof(T);                   // elements per 16-byte vector
    const int lo = max(0, ixb), hi = min(g.IW, ixb + pitch);
    const int r0 = max(0, -iy0), r1 = min(srows, g.IH - iy0);
    const bool vec = (g.IW % VE) == 0 && (g.IS % VE) == 0;
    if (vec && hi > lo && r1 > r0) {
      const int v0 = lo / VE, v1 = (hi + VE - 1) / VE;   // vectors of input columns
      const int nvr = v1 - v0;
      const int total = (r1 - r0) * nvr;
      for (int i0 = threadIdx.x; i0 < total; i0 += 4 * blockDim.x) {
        uint4 buf[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = i0 + u * blockDim.x;
          if (i < total) {
            const int rr = r0 + i / nvr, vv = v0 + i % nvr;
            buf[u] = *reinterpret_cast<const uint4*>(xp + (long long)(iy0 + rr) * g.IW + vv * VE);
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = i0 + u * blockDim.x;
          if (i < total) {
            const int rr = r0 + i / nvr, vv = v0 + i % nvr;
            const T* e = reinterpret_cast<const T*>(&buf[u]);
#pragma unroll
            for (int k = 0; k < VE; ++k) {
              const int ix = vv * VE + k;
              if (ix >= lo && ix < hi) sx[rr * pitch + (ix - ixb)] = to_f32(e[k]);
            }
          }
        }
      }
    } else {
      for (int i = threadIdx.x; i < (r1 - r0) * (hi - lo); i += blockDim.x) {
        const int rr = r0 + i / (hi - lo), ix = lo + i % (hi - lo);
        sx[rr * pitch + (ix - ixb)] = to_f32(xp[(long long)(iy0 + rr) * g.IW + ix]);
      }
    }
  }
  __syncthreads();

  const int tcols = TC / 4;
  const int ty = threadIdx.x / tcols, tx = threadIdx.x - ty * tcols;
  if (ty * 4 >= TR) return;
  const int oy = oy0 + ty * 4, ox = ox0 + tx * 4;
  if (oy >= g.OH || ox >= g.OW) return;
  float acc[4][4];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[r][j] = bias;
  // tile column of output ox + j, tap kx: (ox + j + kx - pW) - ixb = tx*4 + 4 + j + kx
  const float* base = sx + (ty * 4) * pitch + tx * 4 + 4;
#pragma unroll
  for (int ir = 0; ir < 4 + KH - 1; ++ir) {
    float win[WV * 4];
    const float4* rp = reinterpret_cast<const float4*>(base + ir * pitch);
#pragma unroll
    for (int q = 0; q < WV; ++q) {
      const float4 f = rp[q];
      win[4 * q] = f.x; win[4 * q + 1] = f.y; win[4 * q + 2] = f.z; win[4 * q + 3] = f.w;
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int ky = ir - r;
      if (ky < 0 || ky >= KH) continue;
#pragma unroll
      for (int kx = 0; kx < KW; ++kx) {
        const float wv = wr[ky * KW + kx];
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[r][j] = fmaf(win[j + kx], wv, acc[r][j]);
      }
    }
  }
  const long long ybase = (long long)plane * g.P + (long long)oy * g.OW + ox;
  const int nv = min(4, g.OW - ox), nr = min(4, g.OH - oy);
#define FCONV_DW_STORE(ACT) store_block4<ACT, T>(acc, z, y, ybase, g.OW, nr, nv, g.alpha, g.beta)
  FCONV_ACT_SWITCH(g.act, FCONV_DW_STORE)
#undef FCONV_DW_STORE
}


// Persistent variant for planes that fit one tile (OH <= 64, OW <= 64) with stride 1,
// dilation 1: a CTA loops over (image, channel) planes. The zero padding of the fp32
// tile is written once (every plane has the same halo), the next plane's input rows are
// loaded into registers while the current plane is computed, and each thread's Z values
// are requested before its FMA loop so their latency hides behind it. The plane's
// weights sit in shared memory (rows of 8 floats, read as broadcast vectors) rather than
// in registers, so that more CTAs fit on an SM.
template <typename T, int KH, int KW, int MAXV>
__global__ void __launch_bounds__(256) dw_kernel_persistent(ConvGeom g, const T* __restrict__ x,
                                                            const T* __restrict__ w,
                                                            const T* __restrict__ b,
                                                            const T* __restrict__ z,
                                                            T* __restrict__ y, int TR, int TC,
                                                            int pitch, long long planes) {
  ptx::pdl_wait();  // inputs may be the previous kernel's outputs
  ptx::pdl_trigger();
  extern __shared__ float sx[];
  constexpr int WIN = 4 + KW - 1;
  constexpr int WV = (WIN + 3) / 4;
  constexpr int VE = 16 / sizeof(T);
  // rows of the tile: the last block row of threads reads up to row TR + KH - 2 (TR is OH
  // rounded up to a multiple of 4); the weights follow the tile, KH rows of 8 floats
  // Two such buffers alternate between planes: one barrier per plane, after which the
  // threads compute from one buffer while the next plane is written into the other.
  const int srows = TR + KH - 1;
  const int bufsz = srows * pitch + KH * 8;
  const int ixb = -g.pW - 4;                 // input column of tile column 0
  const int nvr = g.IW / VE;                 // 16-byte vectors per input row
  const int nvec = g.IH * nvr;               // per plane
  for (int i = threadIdx.x * 4; i < 2 * bufsz; i += blockDim.x * 4)
    *reinterpret_cast<float4*>(sx + i) = make_float4(0.f, 0.f, 0.f, 0.f);
  const int tcols = TC / 4;
  const int ty = threadIdx.x / tcols, tx = threadIdx.x - ty * tcols;
  const int oy = ty * 4, ox = tx * 4;
  const bool active = oy < g.OH && ox < g.OW;
  const int nv = active ? min(4, g.OW - ox) : 0, nr = active ? min(4, g.OH - oy) : 0;

  uint4 pre[MAXV];
  auto prefetch = [&](long long plane) {
    const T* xp = x + plane * g.IS;
#pragma unroll
    for (int u = 0; u < MAXV; ++u) {
      const int i = threadIdx.x + u * blockDim.x;
      if (i < nvec) pre[u] = *reinterpret_cast<const uint4*>(xp + (long long)i * VE);
    }
  };
  // the prefetched plane's weights and input rows into buffer buf (halo stays zero)
  auto fill = [&](float* buf, long long pl) {
    const int c = (int)(pl % g.C);
    float* sw = buf + srows * pitch;
    for (int i = threadIdx.x; i < KH * 8; i += blockDim.x) {
      const int ky = i >> 3, kx = i & 7;
      sw[i] = kx < KW ? to_f32(w[(long long)c * KH * KW + ky * KW + kx]) : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < MAXV; ++u) {
      const int i = threadIdx.x + u * blockDim.x;
      if (i < nvec) {
        const int iy = i / nvr, c0 = (i - iy * nvr) * VE;
        const T* e = reinterpret_cast<const T*>(&pre[u]);
        float* d = buf + (iy + g.pH) * pitch + (c0 - ixb);
#pragma unroll
        for (int k = 0; k < VE; ++k) d[k] = to_f32(e[k]);
      }
    }
  };
  long long plane = blockIdx.x;
  if (plane < planes) {
    prefetch(plane);
    __syncthreads();  // the zero fill of both buffers is complete
    fill(sx, plane);
    __syncthreads();
    if (plane + gridDim.x < planes) prefetch(plane + gridDim.x);
  }
  for (int k = 0; plane < planes; plane += gridDim.x, k ^= 1) {
    const float* cur = sx + k * bufsz;
    const float* sw = cur + srows * pitch;
    const int c = (int)(plane % g.C);
    const float bias = b ? to_f32(b[c]) : 0.0f;
    const long long obase = plane * g.P + (long long)oy * g.OW + ox;
    // Z is requested before the FMAs and added after them, so its latency overlaps them
    // (whole 4-wide runs: OW % 4 == 0 on this path, nv == 4)
    uint2 zraw[4];  // the four rows' Z, as loaded (f16: 4 values; f32: converted below)
    float4 zf[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      zraw[r] = make_uint2(0u, 0u);
      zf[r] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (z && r < nr) {
        if constexpr (sizeof(T) == 2) zraw[r] = *reinterpret_cast<const uint2*>(z + obase + (long long)r * g.OW);
        else zf[r] = *reinterpret_cast<const float4*>(z + obase + (long long)r * g.OW);
      }
    }
    if (active) {
      float acc[4][4];
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[r][j] = bias;
      const float* base = cur + oy * pitch + ox + 4;
#pragma unroll
      for (int ir = 0; ir < 4 + KH - 1; ++ir) {
        float win[WV * 4];
        const float4* rp = reinterpret_cast<const float4*>(base + ir * pitch);
#pragma unroll
        for (int q = 0; q < WV; ++q) {
          const float4 f = rp[q];
          win[4 * q] = f.x; win[4 * q + 1] = f.y; win[4 * q + 2] = f.z; win[4 * q + 3] = f.w;
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int ky = ir - r;
          if (ky < 0 || ky >= KH) continue;
          float wv[8];
          const float4 w0 = *reinterpret_cast<const float4*>(sw + ky * 8);
          const float4 w1 = *reinterpret_cast<const float4*>(sw + ky * 8 + 4);
          wv[0] = w0.x; wv[1] = w0.y; wv[2] = w0.z; wv[3] = w0.w;
          wv[4] = w1.x; wv[5] = w1.y; wv[6] = w1.z; wv[7] = w1.w;
#pragma unroll
          for (int kx = 0; kx < KW; ++kx)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[r][j] = fmaf(win[j + kx], wv[kx], acc[r][j]);
        }
      }
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        float zr[4];
        if constexpr (sizeof(T) == 2) {
          const __half2 a2 = *reinterpret_cast<const __half2*>(&zraw[r].x);
          const __half2 b2 = *reinterpret_cast<const __half2*>(&zraw[r].y);
          zr[0] = __low2float(a2); zr[1] = __high2float(a2); zr[2] = __low2float(b2); zr[3] = __high2float(b2);
        } else {
          zr[0] = zf[r].x; zr[1] = zf[r].y; zr[2] = zf[r].z; zr[3] = zf[r].w;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[r][j] += zr[j];
      }
#define FCONV_DW_STORE(ACT) store_rows4<ACT, T>(acc, y, obase, g.OW, nr, g.alpha, g.beta)
      FCONV_ACT_SWITCH(g.act, FCONV_DW_STORE)
#undef FCONV_DW_STORE
    }
    const long long next = plane + gridDim.x;
    if (next < planes) fill(sx + (k ^ 1) * bufsz, next);
    __syncthreads();  // next plane staged; everyone is done with this plane's buffer
    if (next + gridDim.x < planes) prefetch(next + gridDim.x);
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
  ptx::pdl_wait();  // inputs may be the previous kernel's outputs
  ptx::pdl_trigger();
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
  const bool unit = g.sW == 1 && g.dW == 1 && g.sH == 1 && g.dH == 1;
  constexpr int VE = 16 / sizeof(T);
  if (unit && g.KH == g.KW && (g.KW == 3 || g.KW == 5 || g.KW == 7) && g.OH <= 64 &&
      g.OW <= 64 && g.OW % 4 == 0 && g.IW % VE == 0 && g.IS % VE == 0 &&
      (long long)g.IH * (g.IW / VE) <= 4LL * ((g.OW + 3) / 4) * ((g.OH + 3) / 4) &&
      g.IH + g.pH <= g.OH + g.KH - 1 && g.IW + g.pW + 4 <= (g.OW + 3) / 4 * 4 + 4 + g.KW + 3) {
    // persistent CTAs; the whole plane is one tile
    const int TC = (g.OW + 3) / 4 * 4;
    const int TR = (g.OH + 3) / 4 * 4;
    const int threads = (TC / 4) * (TR / 4);
    const int pitch = (TC + 4 + g.KW + 3 + 3) / 4 * 4 + 4;
    const size_t smem = 2 * ((size_t)(TR + g.KH - 1) * pitch + (size_t)g.KH * 8) * sizeof(float);
    const long long planes = (long long)g.N * g.C;
    int dev = 0, sms = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
#define FCONV_DW_PERSIST(KV)                                                                    \
  if (g.KW == KV) {                                                                             \
    auto k = dw_kernel_persistent<T, KV, KV, 4>;                                                \
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);           \
    int per_sm = 1;                                                                             \
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, threads, smem);                  \
    long long grid = (long long)sms * (per_sm > 0 ? per_sm : 1);                                \
    if (grid > planes) grid = planes;                                                           \
    if (g.max_ctas > 0 && grid > g.max_ctas) grid = g.max_ctas;                                 \
    return launch_pdl(k, dim3((unsigned)grid), dim3(threads), smem, s, g, x, w, b, z, y, TR, TC, \
                      pitch, planes);                                                           \
  }
    FCONV_DW_PERSIST(3)
    FCONV_DW_PERSIST(5)
    FCONV_DW_PERSIST(7)
#undef FCONV_DW_PERSIST
  }
  if (unit && g.KH == g.KW && (g.KW == 3 || g.KW == 5 || g.KW == 7)) {
    // output tile: TC columns (<= 64, a multiple of 4), TR rows, at most 256 threads
    const int TC = min(64, (g.OW + 3) / 4 * 4);
    int TR = min((g.OH + 3) / 4 * 4, (256 / (TC / 4)) * 4);
    if (TR > 64) TR = 64;
    const int tiles_r = (g.OH + TR - 1) / TR, tiles_c = (g.OW + TC - 1) / TC;
    const int pitch = (TC + 4 + g.KW + 3 + 3) / 4 * 4 + 4;  // vector reads stay in the row
    const size_t smem = (size_t)(TR + g.KH - 1) * pitch * sizeof(float);
    const long long nblk = (long long)g.N * g.C * tiles_r * tiles_c;
    const int threads = (TC / 4) * (TR / 4);
#define FCONV_DW_BLOCK(KV)                                                                     \
  if (g.KW == KV) {                                                                            \
    auto k = dw_kernel_block<T, KV, KV>;                                                       \
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);          \
    return launch_pdl(k, dim3((unsigned)nblk), dim3(threads), smem, s, g, x, w, b, z, y, TR, TC, \
                      tiles_r, tiles_c, pitch);                                                \
  }
    FCONV_DW_BLOCK(3)
    FCONV_DW_BLOCK(5)
    FCONV_DW_BLOCK(7)
#undef FCONV_DW_BLOCK
  }
  auto k = dw_kernel_generic<T>;
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.smem);
  return launch_pdl(k, dim3((unsigned)blocks), dim3(kDwThreads), L.smem, s, g, x, w, b, z, y, L.band,
                    L.bands, L.srows, L.scols);
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
