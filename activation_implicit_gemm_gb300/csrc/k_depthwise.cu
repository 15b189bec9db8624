// Depthwise 2-D FusedConv (C == M == group, one input and one output channel per group)
// on CUDA cores, bandwidth-first: the package's grouped large-kernel route
// (conv2d-grouped-large-w4: a shared input window held in registers, a 4-wide output
// vector per thread, bias seeding the accumulators, f32 accumulation) restated for
// GB300.
//
// Kernels, in the order the host picks them (launch_dw_t):
//   dw_stream_kernel   stride 1, K in {3, 5, 7}, the same-size left pad, rows of X and Y in
//                      whole 4-element vectors: a thread walks 4 output columns down a
//                      whole plane with K rolling accumulator rows (see its comment)
//   dw_tile_kernel     other stride-1 shapes whose X rows TMA can address: persistent,
//                      TMA-staged tiles, TH-row register strips
//   dw_kernel_block    other stride-1 shapes with K in {3, 5, 7}
//   dw_kernel_generic  any stride and dilation: one CTA per (image, channel, band of output
//                      rows) stages the band's input rows, zero-padded, in shared memory as
//                      fp32; each thread makes one output at a time
// All apply bias, residual Z, the activation and the cast to T before the store.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstring>

#include "tc_common.cuh"

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


// Tiled persistent path: stride 1 and dilation 1 on both axes, KH == KW == K known at
// compile time, rows of X that TMA can address (16-byte multiples). The work is a list of
// units (channel c, image n, output tile of THo x TWo), channel-major so that consecutive
// units share their weights. A CTA takes a contiguous range of groups of PP units and
// loops over it with a ring of NS shared-memory stages:
//   - the load warp fills a stage NS groups ahead of the compute: the tile's receptive
//     field of X (positions outside X filled with zeros by TMA, which is the zero padding)
//     and the tile of Z;
//   - thread (unit pp, column group cg, row strip) computes 4 consecutive outputs of TH
//     consecutive rows. Each input row of its receptive field is read once from the box as
//     16 values (f16: four 8-byte loads; f32: four 16-byte loads), converted to f32 and
//     used for every output row it feeds: K x K x 4 x TH FMAs in f32 from K + 3 values per
//     row. The weights stay in registers and are reloaded only when the unit's channel
//     changes (a TMA store of Y from the stage, or weights staged per group, measured
//     slower on the 56 x 56 x 7 x 7 stem shape);
//   - bias seeds the accumulators; + Z, the activation and one rounding to T follow, and
//     the 4 outputs of a row leave as one 8-byte (f16) or 16-byte (f32) store.
// The box starts at the 16-byte boundary at or left of the tile's first input column, so
// the first input column sits OFF = 0..3 elements into a thread's 16-value read; OFF is
// the same for every tile (tiles are multiples of 8 columns wide) and selects one of four
// compiled copies of the FMA block. Every wait is bounded in time; a wait that runs out
// sets the device error word and the CTA leaves after the copies it issued have landed.
constexpr int kDwTileThreads = 256;
constexpr int kDwStages = 3;

struct DwTileArgs {
  int TWo, THo;           // output tile
  int BW, BH;             // input box (elements)
  int a_off;              // box column of the tile's first input column (ox0 - pW)
  int ncg, nstrip, tpu;   // column groups, row strips and threads per unit
  int PP;                 // units per group (computed together)
  int tiles_w, tiles_h;
  long long units, groups;
  int z_tma;              // Z tile loaded by TMA (1) or read from global memory (0)
  int vec_y;              // 4 outputs per row as one vector store (OW % 4 == 0)
  uint32_t xbox_bytes, zbox_bytes;  // bytes of one input box and one Z tile
  uint32_t z_off;         // the Z tile's offset in a unit's slot (128-byte aligned)
  uint32_t unit_bytes, stage_bytes;
  uint32_t bar_off;       // byte offset of the stage barriers
};

// The 16 values at a thread's read position in one box row, K + 3 of them (from OFF on)
// converted to f32.
template <typename T, int K, int OFF>
__device__ __forceinline__ void dw_window(const T* row, float (&win)[K + 3]) {
  constexpr int NQ = (OFF + K + 3 + 3) / 4;  // 4-element groups read
  if constexpr (sizeof(T) == 2) {
    uint2 q[NQ];
#pragma unroll
    for (int i = 0; i < NQ; ++i) q[i] = reinterpret_cast<const uint2*>(row)[i];
    const __half* h = reinterpret_cast<const __half*>(q);
#pragma unroll
    for (int i = 0; i < K + 3; ++i) win[i] = __half2float(h[i + OFF]);
  } else {
    float4 q[NQ];
#pragma unroll
    for (int i = 0; i < NQ; ++i) q[i] = reinterpret_cast<const float4*>(row)[i];
    const float* f = reinterpret_cast<const float*>(q);
#pragma unroll
    for (int i = 0; i < K + 3; ++i) win[i] = f[i + OFF];
  }
}

// acc[o][j] += sum over (ky, kx) of W[ky][kx] * X[strip row o + ky][column j + kx]: every
// box row of the strip's receptive field is read once and feeds up to K output rows.
template <typename T, int K, int TH, int OFF>
__device__ __forceinline__ void dw_strip(const T* box, int BW, const float (&wr)[K * K],
                                         float (&acc)[TH][4]) {
#pragma unroll
  for (int r = 0; r < TH + K - 1; ++r) {
    float win[K + 3];
    dw_window<T, K, OFF>(box + r * BW, win);
    // kx outer: consecutive FMAs update different accumulators (up to 4 x TH in flight)
#pragma unroll
    for (int kx = 0; kx < K; ++kx) {
#pragma unroll
      for (int o = 0; o < TH; ++o) {
        const int ky = r - o;
        if (ky < 0 || ky >= K) continue;
        const float wv = wr[ky * K + kx];
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[o][j] = fmaf(win[j + kx], wv, acc[o][j]);
      }
    }
  }
}

// Half2 row partials (opt-in precision mode, f16 only): for each kernel row the K taps of
// two adjacent outputs are summed with packed f16 FMAs (each rounded once to f16), and the
// row's two partial pairs are then added to the f32 accumulators. Against the f32 path this
// trades K FMAs of error per kernel row (at most K * 2^-11 * sum |x*w| over the row) for
// half the FMA instructions. The pair of outputs (j, j + 1) at tap kx needs the inputs
// (j + kx + OFF, j + kx + OFF + 1): from the 16 halves of the row read as 8 words, an even
// start is one word and an odd start a byte permute of two.
__device__ __forceinline__ uint32_t prmt_b32(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

template <int K, int TH, int OFF>
__device__ __forceinline__ void dw_strip_h2(const __half* box, int BW, const uint32_t (&wh)[K * K],
                                            float (&acc)[TH][4]) {
#pragma unroll
  for (int r = 0; r < TH + K - 1; ++r) {
    uint32_t wv[8];
    const uint2* rp = reinterpret_cast<const uint2*>(box + r * BW);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint2 q = rp[i];
      wv[2 * i] = q.x;
      wv[2 * i + 1] = q.y;
    }
    uint32_t pr[K + 2];  // pr[t] = (x[OFF + t], x[OFF + t + 1])
#pragma unroll
    for (int t = 0; t < K + 2; ++t) {
      const int s0 = OFF + t;
      pr[t] = (s0 % 2 == 0) ? wv[s0 / 2] : prmt_b32(wv[s0 / 2], wv[s0 / 2 + 1], 0x5432u);
    }
#pragma unroll
    for (int o = 0; o < TH; ++o) {
      const int ky = r - o;
      if (ky < 0 || ky >= K) continue;
      __half2 p0 = __hmul2(*reinterpret_cast<const __half2*>(&pr[0]),
                           *reinterpret_cast<const __half2*>(&wh[ky * K]));
      __half2 p1 = __hmul2(*reinterpret_cast<const __half2*>(&pr[2]),
                           *reinterpret_cast<const __half2*>(&wh[ky * K]));
#pragma unroll
      for (int kx = 1; kx < K; ++kx) {
        const __half2 w2 = *reinterpret_cast<const __half2*>(&wh[ky * K + kx]);
        p0 = __hfma2(*reinterpret_cast<const __half2*>(&pr[kx]), w2, p0);
        p1 = __hfma2(*reinterpret_cast<const __half2*>(&pr[kx + 2]), w2, p1);
      }
      const float2 f0 = __half22float2(p0), f1 = __half22float2(p1);
      acc[o][0] += f0.x;
      acc[o][1] += f0.y;
      acc[o][2] += f1.x;
      acc[o][3] += f1.y;
    }
  }
}

// + Z, activation, rounding and the stores of a strip (rows past OH and columns past OW
// are not stored).
template <int ACT, typename T, int TH>
__device__ __forceinline__ void dw_strip_store(const ConvGeom& g, const DwTileArgs& a,
                                               const float (&acc)[TH][4], const T* zs, bool has_z,
                                               const T* __restrict__ z, T* __restrict__ y,
                                               long long obase, int oy, int ox) {
  const int nv = min(4, g.OW - ox);
#pragma unroll
  for (int o = 0; o < TH; ++o) {
    if (oy + o >= g.OH) break;
    const T* zr = zs + o * a.TWo;
    const long long orow = obase + (long long)(oy + o) * g.OW + ox;
    float zv[4] = {0.f, 0.f, 0.f, 0.f};
    if (has_z) {
      if (a.z_tma) {
        if constexpr (sizeof(T) == 2) {
          const uint2 q = *reinterpret_cast<const uint2*>(zr);
          const __half2 lo = *reinterpret_cast<const __half2*>(&q.x);
          const __half2 hi = *reinterpret_cast<const __half2*>(&q.y);
          zv[0] = __low2float(lo); zv[1] = __high2float(lo);
          zv[2] = __low2float(hi); zv[3] = __high2float(hi);
        } else {
          const float4 q = *reinterpret_cast<const float4*>(zr);
          zv[0] = q.x; zv[1] = q.y; zv[2] = q.z; zv[3] = q.w;
        }
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (j < nv) zv[j] = to_f32(z[orow + j]);
      }
    }
    float v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = act_eval<ACT, sizeof(T) == 2>(acc[o][j] + zv[j], g.alpha, g.beta);
    if (a.vec_y && nv == 4) {
      store4(y + orow, v);
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (j < nv) y[orow + j] = from_f32<T>(v[j]);
    }
  }
}

// ------------------------------------------------------------------ column streaming
// dw_stream_kernel: stride 1, dilation 1, K in {3, 5, 7}, rows of X and Y a multiple of 4
// elements. A thread owns 4 adjacent output columns of one (n, c) plane over the plane's
// whole height and walks the input rows top to bottom once: input row r - pH feeds the K
// output rows r - K + 1 .. r, held as K rolling rows of 4 accumulators (slot s meets the
// row with kernel row K - 1 - s). After a row, slot 0 is complete and leaves (+ Z,
// activation, one rounding to T, one vector store); the slots move down by one and the
// last is seeded with the bias. Each thread streams its input rows (4-element vectors,
// zeros outside X, which is the padding) and Z rows through a private ring of asynchronous
// copies into shared memory, kDwStreamAhead - 1 rows ahead of their use, so the loads are
// in flight during the FMAs; no thread reads another's slots, so there is no barrier. The
// loop body is one row (K*K*4 FMAs), small enough for the instruction cache. The tiled
// kernel (below) covers the other shapes.
template <typename T>
struct DwVec;
template <>
struct DwVec<__half> {
  static constexpr uint32_t bytes = 8;
  static __device__ __forceinline__ void copy(uint32_t dst, const void* src, uint32_t n) {
    ptx::cp_async8(dst, src, n);
  }
  static __device__ __forceinline__ void read(uint32_t at, float* f) {
    uint32_t lo, hi;
    asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(lo), "=r"(hi) : "r"(at));
    const __half2 l = *reinterpret_cast<const __half2*>(&lo);
    const __half2 h = *reinterpret_cast<const __half2*>(&hi);
    f[0] = __low2float(l); f[1] = __high2float(l);
    f[2] = __low2float(h); f[3] = __high2float(h);
  }
};
template <>
struct DwVec<float> {
  static constexpr uint32_t bytes = 16;
  static __device__ __forceinline__ void copy(uint32_t dst, const void* src, uint32_t n) {
    ptx::cp_async16(dst, src, n);
  }
  static __device__ __forceinline__ void read(uint32_t at, float* f) {
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(f[0]), "=f"(f[1]), "=f"(f[2]), "=f"(f[3]) : "r"(at));
  }
};

// One CTA of 384 threads per SM (at most): the columns are spread evenly over the SMs
// whichever SMs free up first when the kernel starts behind another one.
constexpr int kDwStreamThreads = 384;
constexpr int kDwStreamAhead = 4;  // rows of X (and Z) in the ring per thread

// 4-element vectors per input row. The ring of one CTA: slot (row % kDwStreamAhead,
// vector q) of thread t at ((slot * (NQ + 1) + q) * kDwStreamThreads + t) * bytes (vector
// q == NQ holds Z), so that a warp's reads of one vector are consecutive.
template <typename T, int K, int OFF>
__host__ __device__ constexpr int dw_stream_nq() { return (OFF + K + 3 + 3) / 4; }

template <typename T, int K, int OFF, int ACT, bool H2>
__device__ __forceinline__ void dw_stream_column(const ConvGeom& g, const T* __restrict__ x,
                                                 const T* __restrict__ w, const T* __restrict__ b,
                                                 const T* __restrict__ z, T* __restrict__ y,
                                                 long long plane, int t, uint32_t ring) {
  using V = DwVec<T>;
  constexpr int NQ = dw_stream_nq<T, K, OFF>();
  constexpr int D = kDwStreamAhead;
  const int c = (int)(plane % g.C);
  float wr[H2 ? 1 : K * K];
  uint32_t wh[H2 ? K * K : 1];  // half2 (w, w) per tap in the half2 mode
  if constexpr (H2) {
#pragma unroll
    for (int i = 0; i < K * K; ++i) {
      const __half2 h2 = __half2half2(*reinterpret_cast<const __half*>(&w[(long long)c * K * K + i]));
      wh[i] = *reinterpret_cast<const uint32_t*>(&h2);
    }
  } else {
#pragma unroll
    for (int i = 0; i < K * K; ++i) wr[i] = to_f32(w[(long long)c * K * K + i]);
  }
  const float bias = b ? to_f32(b[c]) : 0.0f;
  const int ox = 4 * t;
  const int xs = ox - g.pW - OFF;  // column of the first vector (a multiple of 4)
  bool cok[NQ];
#pragma unroll
  for (int q = 0; q < NQ; ++q) cok[q] = xs + 4 * q >= 0 && xs + 4 * q < g.IW;
  const T* xp = x + plane * (long long)g.IH * g.IW;
  const long long ob = plane * (long long)g.OH * g.OW + ox;
  const uint32_t me = ring + (uint32_t)threadIdx.x * V::bytes;
  constexpr uint32_t kStep = kDwStreamThreads * V::bytes;  // one vector of every thread
  const int rows = g.OH + K - 1;
  // step r: input row r - pH, and Z of the output row r - (K - 1) that leaves at step r;
  // zeros (nothing read) outside X, and for Z before the first output row or without Z
  auto issue = [&](int r) {
    const uint32_t slot = me + (uint32_t)((r % D) * (NQ + 1)) * kStep;
    const int ir = r - g.pH;
    const bool rok = r < rows && ir >= 0 && ir < g.IH;
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      const bool ok = rok && cok[q];
      V::copy(slot + (uint32_t)q * kStep,
              ok ? (const void*)(xp + (long long)ir * g.IW + xs + 4 * q) : (const void*)x,
              ok ? V::bytes : 0u);
    }
    const int o = r - (K - 1);
    const bool zok = z != nullptr && r < rows && o >= 0;
    V::copy(slot + (uint32_t)NQ * kStep,
            zok ? (const void*)(z + ob + (long long)o * g.OW) : (const void*)x, zok ? V::bytes : 0u);
    ptx::cp_async_commit();
  };
#pragma unroll
  for (int r = 0; r < D - 1; ++r) issue(r);
  float acc[K][4];
#pragma unroll
  for (int sl = 0; sl < K; ++sl)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[sl][j] = bias;
#pragma unroll 1
  for (int r = 0; r < rows; ++r) {
    issue(r + D - 1);             // D - 1 rows ahead of this one
    ptx::cp_async_wait<D - 1>();  // this step's group has landed
    const uint32_t slot = me + (uint32_t)((r % D) * (NQ + 1)) * kStep;
    if constexpr (H2) {
      // half2 row partials (the tiled kernel's arithmetic, in the same order): per slot and
      // pair of outputs (j, j + 1), the K taps of the slot's kernel row in packed f16 FMAs,
      // then added to the f32 accumulators
      uint32_t wv[2 * NQ];
#pragma unroll
      for (int q = 0; q < NQ; ++q)
        asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];"
                     : "=r"(wv[2 * q]), "=r"(wv[2 * q + 1]) : "r"(slot + (uint32_t)q * kStep));
      uint32_t pr[K + 2];  // pr[u] = (x[OFF + u], x[OFF + u + 1])
#pragma unroll
      for (int u = 0; u < K + 2; ++u) {
        const int s0 = OFF + u;
        pr[u] = (s0 % 2 == 0) ? wv[s0 / 2] : prmt_b32(wv[s0 / 2], wv[s0 / 2 + 1], 0x5432u);
      }
#pragma unroll
      for (int sl = 0; sl < K; ++sl) {
        const int ky = K - 1 - sl;
        __half2 p0 = __hmul2(*reinterpret_cast<const __half2*>(&pr[0]),
                             *reinterpret_cast<const __half2*>(&wh[ky * K]));
        __half2 p1 = __hmul2(*reinterpret_cast<const __half2*>(&pr[2]),
                             *reinterpret_cast<const __half2*>(&wh[ky * K]));
#pragma unroll
        for (int kx = 1; kx < K; ++kx) {
          const __half2 w2 = *reinterpret_cast<const __half2*>(&wh[ky * K + kx]);
          p0 = __hfma2(*reinterpret_cast<const __half2*>(&pr[kx]), w2, p0);
          p1 = __hfma2(*reinterpret_cast<const __half2*>(&pr[kx + 2]), w2, p1);
        }
        const float2 f0 = __half22float2(p0), f1 = __half22float2(p1);
        acc[sl][0] += f0.x;
        acc[sl][1] += f0.y;
        acc[sl][2] += f1.x;
        acc[sl][3] += f1.y;
      }
    } else {
      float win[4 * NQ];
#pragma unroll
      for (int q = 0; q < NQ; ++q) V::read(slot + (uint32_t)q * kStep, win + 4 * q);
#pragma unroll
      for (int kx = 0; kx < K; ++kx)
#pragma unroll
        for (int sl = 0; sl < K; ++sl) {
          const float wv = wr[(K - 1 - sl) * K + kx];
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[sl][j] = fmaf(win[OFF + j + kx], wv, acc[sl][j]);
        }
    }
    const int o = r - (K - 1);  // the output row slot 0 completes now
    if (o >= 0) {
      float zv[4];
      V::read(slot + (uint32_t)NQ * kStep, zv);
      float v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        v[j] = act_eval<ACT, sizeof(T) == 2>(acc[0][j] + zv[j], g.alpha, g.beta);
      store4(y + ob + (long long)o * g.OW, v);
    }
#pragma unroll
    for (int sl = 0; sl < K - 1; ++sl)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[sl][j] = acc[sl + 1][j];
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[K - 1][j] = bias;
  }
  ptx::cp_async_wait<0>();  // the ring's last (empty) groups, before the slots are reused
}

template <typename T, int K, int OFF, bool H2>
__global__ void __launch_bounds__(kDwStreamThreads, 1)
    dw_stream_kernel(const ConvGeom g, int tpp, long long nthr, const T* __restrict__ x,
                     const T* __restrict__ w, const T* __restrict__ b, const T* __restrict__ z,
                     T* __restrict__ y) {
  extern __shared__ __align__(16) uint8_t dws[];
  const uint32_t ring = ptx::smem_addr(dws);
  ptx::pdl_wait();  // inputs may be the previous kernel's outputs
  ptx::pdl_trigger();
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x; gid < nthr; gid += stride) {
    const long long plane = gid / tpp;
    const int t = (int)(gid - plane * tpp);
#define FCONV_DW_STREAM(ACT) dw_stream_column<T, K, OFF, ACT, H2>(g, x, w, b, z, y, plane, t, ring)
    FCONV_ACT_SWITCH(g.act, FCONV_DW_STREAM)
#undef FCONV_DW_STREAM
  }
}

// Unit u -> (channel, image, tile row, tile column).
struct DwUnit {
  int c, n, th, tw;
};
__device__ __forceinline__ DwUnit dw_unit(const DwTileArgs& a, int N, int u) {
  const int tiles = a.tiles_w * a.tiles_h;
  DwUnit r;
  const int nt = N * tiles;
  r.c = u / nt;
  const int rem = u - r.c * nt;
  r.n = rem / tiles;
  const int t = rem - r.n * tiles;
  r.th = t / a.tiles_w;
  r.tw = t - r.th * a.tiles_w;
  return r;
}

template <typename T, int K, int TH, bool H2>
__global__ void __launch_bounds__(kDwTileThreads, 2)
    dw_tile_kernel(const ConvGeom g, const DwTileArgs a, const T* __restrict__ w,
                   const T* __restrict__ b, const T* __restrict__ z, T* __restrict__ y,
                   const __grid_constant__ CUtensorMap tx, const __grid_constant__ CUtensorMap tz) {
  extern __shared__ __align__(1024) uint8_t dsm[];
  const uint32_t sbase = ptx::smem_addr(dsm);
  const uint32_t full = sbase + a.bar_off;             // NS barriers: the stage is filled
  const uint32_t empty = full + 8 * kDwStages;          // NS barriers: the compute warps are done
  volatile int* abort_flag = reinterpret_cast<volatile int*>(dsm + a.bar_off + 16 * kDwStages);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cwarps = (a.PP * a.tpu + 31) >> 5;          // compute warps; the next one loads
  const int per = (int)((a.groups + gridDim.x - 1) / gridDim.x);
  const int q0 = (int)blockIdx.x * per;
  const int q1 = (int)min(a.groups, (long long)q0 + per);
  if (tid == 0) {
    for (int s = 0; s < kDwStages; ++s) {
      ptx::mbar_init(full + 8 * s, 1);
      ptx::mbar_init(empty + 8 * s, (uint32_t)cwarps);
    }
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  ptx::pdl_wait();  // inputs may be the previous kernel's outputs
  ptx::pdl_trigger();

  if (warp == cwarps) {
    // ============================================================== load warp
    if (lane == 0) {
      ptx::prefetch_tmap(&tx);
      if (a.z_tma) ptx::prefetch_tmap(&tz);
      int it = 0;
      for (int q = q0; q < q1; ++q, ++it) {
        const int s = it % kDwStages;
        const uint32_t phase = (uint32_t)(it / kDwStages) & 1u;
        if (!bounded_wait(empty + 8 * s, phase ^ 1u, abort_flag)) {
          // what was issued lands before the CTA leaves
          for (int k = 1; k < kDwStages && it - k >= 0; ++k)
            drain_wait(full + 8 * ((it - k) % kDwStages), (uint32_t)((it - k) / kDwStages) & 1u);
          break;
        }
        const uint32_t bar = full + 8 * s;
        const int ubeg = q * a.PP;
        const int nu = min(a.PP, (int)(a.units - ubeg));
        ptx::mbar_arrive_expect_tx(bar, (uint32_t)nu * (a.xbox_bytes + (a.z_tma ? a.zbox_bytes : 0u)));
        for (int pp = 0; pp < nu; ++pp) {
          const DwUnit un = dw_unit(a, g.N, ubeg + pp);
          const int plane = un.n * g.C + un.c;
          const int ox0 = un.tw * a.TWo, oy0 = un.th * a.THo;
          const uint32_t dst = sbase + (uint32_t)s * a.stage_bytes + (uint32_t)pp * a.unit_bytes;
          ptx::tma_load_3d(dst, &tx, ox0 - g.pW - a.a_off, oy0 - g.pH, plane, bar);
          if (a.z_tma) ptx::tma_load_3d(dst + a.z_off, &tz, ox0, oy0, plane, bar);
        }
      }
    }
    return;
  }
  if (warp > cwarps) return;

  // ================================================================ compute warps
  const int pp = tid / a.tpu, lt = tid - pp * a.tpu;
  const int cg = lt % a.ncg, strip = lt / a.ncg;
  const int off = a.a_off & 3;
  int wc = -1;
  float wr[H2 ? 1 : K * K];
  uint32_t wh[H2 ? K * K : 1];  // half2 (w, w) per tap in the half2 mode
  float bias = 0.0f;
#pragma unroll
  for (int i = 0; i < (H2 ? 1 : K * K); ++i) wr[i] = 0.0f;
#pragma unroll
  for (int i = 0; i < (H2 ? K * K : 1); ++i) wh[i] = 0u;
  int it = 0;
  for (int q = q0; q < q1; ++q, ++it) {
    const int s = it % kDwStages;
    const uint32_t phase = (uint32_t)(it / kDwStages) & 1u;
    if (!bounded_wait(full + 8 * s, phase, abort_flag)) break;
    const int u = q * a.PP + pp;
    if (pp < a.PP && u < a.units) {
      const DwUnit un = dw_unit(a, g.N, u);
      const int ox = un.tw * a.TWo + 4 * cg, oy = un.th * a.THo + strip * TH;
      if (ox < g.OW && oy < g.OH) {
        if (un.c != wc) {
          wc = un.c;
          if constexpr (H2) {
#pragma unroll
            for (int i = 0; i < K * K; ++i) {
              const __half2 h2 = __half2half2(*reinterpret_cast<const __half*>(&w[(long long)un.c * K * K + i]));
              wh[i] = *reinterpret_cast<const uint32_t*>(&h2);
            }
          } else {
#pragma unroll
            for (int i = 0; i < K * K; ++i) wr[i] = to_f32(w[(long long)un.c * K * K + i]);
          }
          bias = b ? to_f32(b[un.c]) : 0.0f;
        }
        const uint8_t* unit = dsm + (size_t)s * a.stage_bytes + (size_t)pp * a.unit_bytes;
        const T* xb = reinterpret_cast<const T*>(unit) + (strip * TH) * a.BW + 4 * cg + (a.a_off & ~3);
        float acc[TH][4];
#pragma unroll
        for (int o = 0; o < TH; ++o)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[o][j] = bias;
        if constexpr (H2) {
          const __half* xh = reinterpret_cast<const __half*>(xb);
          switch (off) {
            case 0: dw_strip_h2<K, TH, 0>(xh, a.BW, wh, acc); break;
            case 1: dw_strip_h2<K, TH, 1>(xh, a.BW, wh, acc); break;
            case 2: dw_strip_h2<K, TH, 2>(xh, a.BW, wh, acc); break;
            default: dw_strip_h2<K, TH, 3>(xh, a.BW, wh, acc); break;
          }
        } else {
          switch (off) {
            case 0: dw_strip<T, K, TH, 0>(xb, a.BW, wr, acc); break;
            case 1: dw_strip<T, K, TH, 1>(xb, a.BW, wr, acc); break;
            case 2: dw_strip<T, K, TH, 2>(xb, a.BW, wr, acc); break;
            default: dw_strip<T, K, TH, 3>(xb, a.BW, wr, acc); break;
          }
        }
        const T* zs = reinterpret_cast<const T*>(unit + a.z_off) + (strip * TH) * a.TWo + 4 * cg;
        const long long obase = ((long long)un.n * g.C + un.c) * g.P;
#define FCONV_DW_TILE_STORE(ACT) \
  dw_strip_store<ACT, T, TH>(g, a, acc, zs, z != nullptr, z, y, obase, oy, ox)
        FCONV_ACT_SWITCH(g.act, FCONV_DW_TILE_STORE)
#undef FCONV_DW_TILE_STORE
      }
    }
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(empty + 8 * s);  // this warp is done with stage s
  }
}

struct DwTilePlan {
  bool ok;
  int TH;
  DwTileArgs a;
  size_t smem;
};

DwTilePlan dw_tile_plan(const ConvGeom& g) {
  DwTilePlan p{};
  p.ok = false;
  const int K = g.KW;
  if (!(g.Cg == 1 && g.Mg == 1 && g.KD == 1 && g.ID == 1 && g.OD == 1)) return p;
  if (!(g.sW == 1 && g.dW == 1 && g.sH == 1 && g.dH == 1 && g.KH == K)) return p;
  if (K != 3 && K != 5 && K != 7) return p;
  const int es = g.dtype == FCONV_F16 ? 2 : 4;
  const int xal = 16 / es;
  if ((g.IW * es) % 16 != 0) return p;  // rows of X must be TMA-addressable
  DwTileArgs& a = p.a;
  a.TWo = imin(64, (g.OW + 7) / 8 * 8);
  a.a_off = ((-g.pW) % xal + xal) % xal;
  a.BW = (a.TWo + (a.a_off & ~3) + 12 + xal - 1) / xal * xal;
  a.ncg = a.TWo / 4;
  a.tiles_w = (g.OW + a.TWo - 1) / a.TWo;
  // rows per thread and units per group: the fewest issued FMA and load instructions,
  // counting the idle lanes of partly filled warps and the rows past OH
  double best = 0.0;
  const int ths[3] = {8, 7, 4};
  for (int th : ths) {
    const int tho = imin((g.OH + th - 1) / th * th, (64 / th) * th);
    const int nstrip = tho / th;
    const int tpu = a.ncg * nstrip;
    if (tpu > kDwTileThreads - 32) continue;
    const long long units = (long long)g.N * g.C * ((g.OH + tho - 1) / tho) * a.tiles_w;
    for (int pp = 1; (pp * tpu + 31) / 32 * 32 + 32 <= kDwTileThreads && pp <= 8; ++pp) {
      const long long warps = (pp * tpu + 31) / 32;
      const double cost = (double)((units + pp - 1) / pp) * (double)warps *
                          (double)(th * K * K * 4 + (th + K - 1) * 8);
      if (!p.ok || cost < best) {
        best = cost;
        p.ok = true;
        p.TH = th;
        a.THo = tho;
        a.nstrip = nstrip;
        a.tpu = tpu;
        a.PP = pp;
        a.units = units;
      }
    }
  }
  if (!p.ok) return p;
  a.tiles_h = (g.OH + a.THo - 1) / a.THo;
  a.groups = (a.units + a.PP - 1) / a.PP;
  a.BH = a.THo + K - 1;
  a.z_tma = (g.OW * es) % 16 == 0 ? 1 : 0;
  a.vec_y = g.OW % 4 == 0 ? 1 : 0;
  a.xbox_bytes = (uint32_t)(a.BW * a.BH * es);
  a.zbox_bytes = (uint32_t)(a.TWo * a.THo * es);
  // a unit's slot: the input box, then the Z tile
  a.z_off = (a.xbox_bytes + 127u) & ~127u;
  a.unit_bytes = a.z_off + (a.z_tma ? (a.zbox_bytes + 127u) & ~127u : 0u);
  a.stage_bytes = (uint32_t)a.PP * a.unit_bytes;
  a.bar_off = (uint32_t)kDwStages * a.stage_bytes;
  p.smem = (size_t)a.bar_off + 16 * kDwStages + 16;
  if (p.smem > 200 * 1024 || a.units > 0x7fffffffLL) p.ok = false;
  return p;
}

template <typename T>
int launch_dw_tile(const ConvGeom& g, const DwTilePlan& p, const ConvArgs& args, cudaStream_t s) {
  EncodeTiledFn enc = tensor_map_encoder();
  if (!enc) return (int)cudaErrorNotSupported;
  const DwTileArgs& a = p.a;
  const cuuint64_t es = sizeof(T);
  const CUtensorMapDataType dt = sizeof(T) == 2 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const cuuint32_t est[3] = {1, 1, 1};
  CUtensorMap tx, tz;
  std::memset(&tx, 0, sizeof(tx));
  std::memset(&tz, 0, sizeof(tz));
  auto encode = [&](CUtensorMap* m, const void* ptr, cuuint64_t d0, cuuint64_t d1, cuuint32_t b0,
                    cuuint32_t b1) {
    const cuuint64_t dims[3] = {d0, d1, (cuuint64_t)g.N * g.C};
    const cuuint64_t str[2] = {d0 * es, d0 * d1 * es};
    const cuuint32_t box[3] = {b0, b1, 1};
    return enc(m, dt, 3, const_cast<void*>(ptr), dims, str, box, est, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  };
  if (!encode(&tx, args.x, (cuuint64_t)g.IW, (cuuint64_t)g.IH, (cuuint32_t)a.BW, (cuuint32_t)a.BH))
    return (int)cudaErrorInvalidValue;
  DwTileArgs aa = a;
  if (aa.z_tma && args.z) {
    if (!encode(&tz, args.z, (cuuint64_t)g.OW, (cuuint64_t)g.OH, (cuuint32_t)a.TWo, (cuuint32_t)a.THo))
      return (int)cudaErrorInvalidValue;
  } else {
    aa.z_tma = 0;  // nothing to load
  }
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int threads = (a.PP * a.tpu + 31) / 32 * 32 + 32;  // compute warps + the load warp
  const bool h2 = g.precision == FCONV_PRECISION_HALF2_ROWS;
#define FCONV_DW_TILE(KV, THV)                                                                  \
  if (g.KW == KV && p.TH == THV) {                                                              \
    auto k = h2 ? dw_tile_kernel<T, KV, THV, sizeof(T) == 2> : dw_tile_kernel<T, KV, THV, false>; \
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,         \
                                         (int)p.smem);                                          \
    if (e != cudaSuccess) return (int)e;                                                        \
    int per_sm = 1;                                                                             \
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, threads, p.smem);                 \
    long long grid = (long long)sms * (per_sm > 0 ? per_sm : 1);                                \
    if (grid > a.groups) grid = a.groups;                                                       \
    if (g.max_ctas > 0 && grid > g.max_ctas) grid = g.max_ctas;                                 \
    return launch_pdl(k, dim3((unsigned)grid), dim3(threads), p.smem, s, g, aa,                 \
                      (const T*)args.w, (const T*)args.b, (const T*)args.z, (T*)args.y, tx, tz); \
  }
  FCONV_DW_TILE(3, 8) FCONV_DW_TILE(3, 7) FCONV_DW_TILE(3, 4)
  FCONV_DW_TILE(5, 8) FCONV_DW_TILE(5, 7) FCONV_DW_TILE(5, 4)
  FCONV_DW_TILE(7, 8) FCONV_DW_TILE(7, 7) FCONV_DW_TILE(7, 4)
#undef FCONV_DW_TILE
  return (int)cudaErrorInvalidValue;
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

// The column-streaming kernel takes stride 1, dilation 1, K in {3, 5, 7} with the left pad
// of a same-size conv modulo 4 ((K - 1) / 2, so that one vector offset per K is compiled),
// rows of X and Y that are whole 4-element vectors, and vector-aligned X, Z and Y, in the
// default precision or (f16) the half2 mode.
bool dw_stream_ok(const ConvGeom& g) {
  if (!(g.Cg == 1 && g.Mg == 1 && g.KD == 1 && g.ID == 1 && g.OD == 1)) return false;
  if (!(g.sW == 1 && g.dW == 1 && g.sH == 1 && g.dH == 1 && g.KH == g.KW)) return false;
  if (g.KW != 3 && g.KW != 5 && g.KW != 7) return false;
  if ((g.pW - (g.KW - 1) / 2) % 4 != 0) return false;
  if (g.precision != FCONV_PRECISION_DEFAULT &&
      !(g.precision == FCONV_PRECISION_HALF2_ROWS && g.dtype == FCONV_F16))
    return false;
  if (g.N < 1 || g.C < 1 || g.OH < 1 || g.OW < 4) return false;
  return g.IW % 4 == 0 && g.OW % 4 == 0 && (long long)g.N * g.C * (g.OW / 4) < 0x7fffffffLL * 128LL;
}

bool vec_aligned(const void* p, size_t bytes) { return p == nullptr || ((uintptr_t)p % bytes) == 0; }

template <typename T>
int launch_dw_stream(const ConvGeom& g, const ConvArgs& a, cudaStream_t s) {
  const int tpp = g.OW / 4;
  const long long nthr = (long long)g.N * g.C * tpp;
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long grid = (nthr + kDwStreamThreads - 1) / kDwStreamThreads;
  if (grid > sms) grid = sms;
  if (g.max_ctas > 0 && grid > g.max_ctas) grid = g.max_ctas;
  const int off = ((-g.pW) % 4 + 4) % 4;
  const bool h2 = g.precision == FCONV_PRECISION_HALF2_ROWS;
#define FCONV_DW_STREAM_K(KV, OV)                                                              \
  if (g.KW == KV && off == OV) {                                                               \
    auto k = h2 ? dw_stream_kernel<T, KV, OV, sizeof(T) == 2> : dw_stream_kernel<T, KV, OV, false>; \
    const size_t smem = (size_t)kDwStreamAhead * (dw_stream_nq<T, KV, OV>() + 1) *             \
                        kDwStreamThreads * DwVec<T>::bytes;                                    \
    const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,  \
                                               (int)smem);                                       \
    if (e != cudaSuccess) return (int)e;                                                        \
    return launch_pdl(k, dim3((unsigned)grid), dim3(kDwStreamThreads), smem, s, g, tpp, nthr,   \
                      (const T*)a.x, (const T*)a.w, (const T*)a.b, (const T*)a.z, (T*)a.y);     \
  }
  FCONV_DW_STREAM_K(3, 3) FCONV_DW_STREAM_K(5, 2) FCONV_DW_STREAM_K(7, 1)
#undef FCONV_DW_STREAM_K
  return (int)cudaErrorInvalidValue;
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
  if (dw_stream_ok(g) && vec_aligned(a.x, 4 * sizeof(T)) && vec_aligned(a.z, 4 * sizeof(T)) &&
      vec_aligned(a.y, 4 * sizeof(T)))
    return launch_dw_stream<T>(g, a, s);
  {
    const DwTilePlan tp = dw_tile_plan(g);
    if (tp.ok) return launch_dw_tile<T>(g, tp, a, s);
    if (g.precision != FCONV_PRECISION_DEFAULT) return (int)cudaErrorInvalidValue;
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

bool depthwise_half2_supported(const ConvGeom& g) {
  return g.dtype == FCONV_F16 && depthwise_supported(g) && dw_tile_plan(g).ok;
}

int read_and_clear_dw_error(void* stream, unsigned* value) {
  return read_and_clear_tc_error((cudaStream_t)stream, value);
}

int launch_depthwise(const ConvGeom& g, const ConvArgs& a, void* stream) {
  cudaStream_t s = (cudaStream_t)stream;
  if (g.dtype == FCONV_F16) return launch_dw_t<__half>(g, a, s);
  return launch_dw_t<float>(g, a, s);
}

}  // namespace fconv
