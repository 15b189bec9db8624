// Transposed FusedConv, Y = act(convT(X, W) + B + Z), in gather form (ExecuTorch WebGPU PR
// #20849, conv_transpose2d.wgsl: "for each tap (kh, kw) an input row contributes only when
// (oh + pH - kh*dH) is divisible by sH and in range; weight is read in the un-flipped torch
// transposed layout [IC, OC/groups, KH, KW]"), for 1-3 spatial dims, any group, fp16 or
// fp32 with f32 accumulation. W is (C, M/group, kernel...).
//
// Along each axis an output o receives input i through tap k when o + pad = i*s + k*d.
// Outputs with the same o mod s (a stride phase) take the same taps, so the work is laid
// out phase-major along w: a warp computes 32 outputs o_w = ow0 + q*sW + phase (q = lane)
// of one output row, and every lane of the warp tests the same taps. A CTA owns an output
// tile of TD x TH rows x 32*sW columns of one image, one group and MB output channels
// (MB = 1..16 in registers per thread, for two segments), and walks the group's input channels in chunks of
// CC: the tile's receptive field of X (f32, zero outside X) and the chunk's weights
// ([c][tap][m], f32) go to shared memory; then each thread, for every tap valid for its
// phase and row, reads one input value per channel and does MB FMAs with the weights read
// as broadcast 16-byte vectors. The epilogue adds B and Z, applies the activation and
// rounds once to T; a warp's stores of one channel are 32 outputs sW apart.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "epilogue.cuh"
#include "fastdiv.cuh"
#include "fconv_internal.h"
#include "ptx.cuh"

namespace fconv {
namespace {

constexpr int kTrThreads = 256;
constexpr int kTrWarps = kTrThreads / 32;
constexpr size_t kTrSmemBudget = 96 * 1024;
constexpr int kTrSegs = 2;  // (row, w phase) segments a warp holds at once
constexpr int kTrMaxTaps = 128;  // kernels up to this many taps use per-warp tap lists

struct TrArgs {
  int TD, TH;              // output rows of a tile (depth, height)
  int TW;                  // output columns of a tile: 32 * sW
  int nTd, nTh, nTw;       // tiles per axis
  int MB, nmb;             // output channels per CTA and channel blocks per group
  int CC;                  // input channels per shared-memory chunk
  int BD, BH, BW;          // staged input box (positions per axis)
  int KV;
  FastDiv fd_kv, fd_bh, fd_brows;  // division by KV, BH and BD * BH
};

// floor(a / b) for b > 0
__device__ __forceinline__ int fdiv(int a, int b) {
  const int q = a / b;
  return (a % b != 0 && a < 0) ? q - 1 : q;
}

template <typename T, int MB>
__global__ void __launch_bounds__(kTrThreads, 2) convt_kernel(const ConvGeom g, const TrArgs a,
                                                           const T* __restrict__ x,
                                                           const T* __restrict__ w,
                                                           const T* __restrict__ b,
                                                           const T* __restrict__ z,
                                                           T* __restrict__ y) {
  extern __shared__ __align__(16) float tsm[];
  ptx::pdl_wait();  // inputs may be the previous kernel's outputs
  ptx::pdl_trigger();
  // the block: (tile w, tile h, tile d, channel block, group, image)
  long long blk = blockIdx.x;
  const int tw = (int)(blk % a.nTw); blk /= a.nTw;
  const int th = (int)(blk % a.nTh); blk /= a.nTh;
  const int td = (int)(blk % a.nTd); blk /= a.nTd;
  const int mb = (int)(blk % a.nmb); blk /= a.nmb;
  const int grp = (int)(blk % g.G);
  const int n = (int)(blk / g.G);
  const int ow0 = tw * a.TW, oh0 = th * a.TH, od0 = td * a.TD;
  const int m0 = mb * MB;  // first output channel of the block within the group
  // the lowest input index each axis can reach from this tile
  const int iw0 = fdiv(ow0 + g.pW - (g.KW - 1) * g.dW, g.sW);
  const int ih0 = fdiv(oh0 + g.pH - (g.KH - 1) * g.dH, g.sH);
  const int id0 = fdiv(od0 + g.pD - (g.KD - 1) * g.dD, g.sD);
  const int box = a.BD * a.BH * a.BW;
  float* sx = tsm;                                 // [CC][BD][BH][BW]
  float* sw = tsm + (((size_t)a.CC * box + 3) & ~(size_t)3);  // [CC][KV][MB], 16-byte aligned
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int segs = a.TD * a.TH * g.sW;             // (row, w phase) segments of the tile
  const int nseg = (segs + kTrWarps - 1) / kTrWarps;

  // The taps valid for each of the warp's segments and their offsets in the staged box
  // (for lane 0; lane l reads l positions further), computed once: they do not depend on
  // the channel chunk. Taps are uniform across the warp (one w phase per segment).
  int2* tl = reinterpret_cast<int2*>(sw + (((size_t)a.CC * a.KV * MB + 3) & ~(size_t)3));
  int ntap[kTrSegs];
#pragma unroll
  for (int s4 = 0; s4 < kTrSegs; ++s4) {
    ntap[s4] = 0;
    const int seg = warp + s4 * kTrWarps;
    if (s4 >= nseg || seg >= segs) continue;
    const int ph = seg % g.sW, row = seg / g.sW;
    const int oh = oh0 + row % a.TH, od = od0 + row / a.TH;
    if (od >= g.OD || oh >= g.OH) continue;
    int2* list = tl + (size_t)(warp * kTrSegs + s4) * a.KV;
    int cnt = 0;
    for (int k = 0; k < a.KV; ++k) {
      const int kx = k % g.KW, ky = (k / g.KW) % g.KH, kz = k / (g.KW * g.KH);
      const int tz = od + g.pD - kz * g.dD - id0 * g.sD;  // >= 0 by construction
      const int ty = oh + g.pH - ky * g.dH - ih0 * g.sH;
      const int tx = ow0 + ph + g.pW - kx * g.dW - iw0 * g.sW;  // lane 0
      if (tz % g.sD || ty % g.sH || tx % g.sW) continue;
      if (lane == 0)
        list[cnt] = make_int2(k * MB, ((tz / g.sD) * a.BH + ty / g.sH) * a.BW + tx / g.sW);
      ++cnt;
    }
    ntap[s4] = cnt;
  }
  __syncwarp();

  float acc[kTrSegs][MB];
#pragma unroll
  for (int s4 = 0; s4 < kTrSegs; ++s4)
#pragma unroll
    for (int m = 0; m < MB; ++m) acc[s4][m] = 0.0f;

  for (int c0 = 0; c0 < g.Cg; c0 += a.CC) {
    const int cc_n = min(a.CC, g.Cg - c0);
    __syncthreads();  // the previous chunk is consumed
    // the receptive field of the chunk's channels, zero outside X
    const T* xg = x + ((long long)n * g.C + (long long)grp * g.Cg + c0) * g.IS;
    const int brows = a.BD * a.BH;
    const int nrow = cc_n * brows;
    // eight rows per warp in flight: all loads of a batch are issued before its stores
    for (int r0 = warp; r0 < nrow; r0 += kTrWarps * 8) {
      for (int bx0 = 0; bx0 < a.BW; bx0 += 32) {
        const int bx = bx0 + lane;
        const int ix = iw0 + bx;
        const bool col_in = bx < a.BW && ix >= 0 && ix < g.IW;
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int r = r0 + u * kTrWarps;
          v[u] = 0.0f;
          if (r < nrow && col_in) {
            uint32_t c, rr, bz, by;
            fast_divmod((uint32_t)r, a.fd_brows, c, rr);
            fast_divmod(rr, a.fd_bh, bz, by);
            const int iy = ih0 + by, iz = id0 + bz;
            if (iy >= 0 && iy < g.IH && iz >= 0 && iz < g.ID)
              v[u] = to_f32(xg[(long long)c * g.IS + ((long long)iz * g.IH + iy) * g.IW + ix]);
          }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int r = r0 + u * kTrWarps;
          if (r < nrow && bx < a.BW) sx[(size_t)r * a.BW + bx] = v[u];
        }
      }
    }
    // the chunk's weights: W[c][m][tap] -> sw[c][tap][m], zero past the group's channels;
    // eight loads per thread in flight
    const int nwt = cc_n * a.KV * MB;
    for (int e0 = threadIdx.x; e0 < nwt; e0 += kTrThreads * 8) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int e = e0 + u * kTrThreads;
        v[u] = 0.0f;
        if (e < nwt) {
          const int m = e % MB;  // MB is a power of two
          uint32_t c, k;
          fast_divmod((uint32_t)(e / MB), a.fd_kv, c, k);
          const int mm = m0 + m;
          if (mm < g.Mg)
            v[u] = to_f32(w[((long long)(grp * g.Cg + c0 + (int)c) * g.Mg + mm) * a.KV + (int)k]);
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int e = e0 + u * kTrThreads;
        if (e < nwt) sw[e] = v[u];
      }
    }
    __syncthreads();
    // the warp's segments, unrolled so that acc stays in registers
#pragma unroll
    for (int s4 = 0; s4 < kTrSegs; ++s4) {
      const int seg = warp + s4 * kTrWarps;
      if (s4 >= nseg || seg >= segs) continue;
      const int2* list = tl + (size_t)(warp * kTrSegs + s4) * a.KV;
      for (int t = 0; t < ntap[s4]; ++t) {
        const int2 e = list[t];
        const float* xs = sx + e.y + lane;
        const float* ws = sw + e.x;
        const size_t wstep = (size_t)a.KV * MB;
        int c = 0;
        for (; c + 4 <= cc_n; c += 4) {
          float xv[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) xv[u] = xs[(size_t)(c + u) * box];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float* wc = ws + (size_t)(c + u) * wstep;
            if constexpr (MB % 4 == 0) {
#pragma unroll
              for (int q = 0; q < MB / 4; ++q) {
                const float4 wv = reinterpret_cast<const float4*>(wc)[q];
                acc[s4][4 * q] = fmaf(xv[u], wv.x, acc[s4][4 * q]);
                acc[s4][4 * q + 1] = fmaf(xv[u], wv.y, acc[s4][4 * q + 1]);
                acc[s4][4 * q + 2] = fmaf(xv[u], wv.z, acc[s4][4 * q + 2]);
                acc[s4][4 * q + 3] = fmaf(xv[u], wv.w, acc[s4][4 * q + 3]);
              }
            } else {
#pragma unroll
              for (int m = 0; m < MB; ++m) acc[s4][m] = fmaf(xv[u], wc[m], acc[s4][m]);
            }
          }
        }
        for (; c < cc_n; ++c) {
          const float xv = xs[(size_t)c * box];
          const float* wc = ws + (size_t)c * wstep;
#pragma unroll
          for (int m = 0; m < MB; ++m) acc[s4][m] = fmaf(xv, wc[m], acc[s4][m]);
        }
      }
    }
  }
  // epilogue: the segment's Z values are all requested before the first store
#pragma unroll
  for (int s4 = 0; s4 < kTrSegs; ++s4) {
    const int seg = warp + s4 * kTrWarps;
    if (s4 >= nseg || seg >= segs) continue;
    const int ph = seg % g.sW, row = seg / g.sW;
    const int oh = oh0 + row % a.TH, od = od0 + row / a.TH;
    const int ow = ow0 + lane * g.sW + ph;
    if (od >= g.OD || oh >= g.OH || ow >= g.OW) continue;
    const long long pix = ((long long)od * g.OH + oh) * g.OW + ow;
    const long long obase = ((long long)n * g.M + grp * g.Mg + m0) * g.P + pix;
    float zv[MB];
#pragma unroll
    for (int m = 0; m < MB; ++m)
      zv[m] = (z && m0 + m < g.Mg) ? to_f32(z[obase + (long long)m * g.P]) : 0.0f;
#pragma unroll
    for (int m = 0; m < MB; ++m) {
      if (m0 + m < g.Mg) {
        float v = acc[s4][m] + zv[m];
        if (b) v += to_f32(b[grp * g.Mg + m0 + m]);
        y[obase + (long long)m * g.P] = from_f32<T>(apply_act(g.act, v, g.alpha, g.beta));
      }
    }
  }
}

struct TrPlan {
  bool ok;
  TrArgs a;
  size_t smem;
  long long blocks;
};

int mb_of(int Mg) {
  static const int inst[] = {1, 2, 4, 8, 16};
  for (int v : inst)
    if (Mg <= v) return v;
  return 16;
}

TrPlan tr_plan(const ConvGeom& g) {
  TrPlan p{};
  p.ok = false;
  TrArgs& a = p.a;
  a.KV = g.KD * g.KH * g.KW;
  a.MB = mb_of(g.Mg);
  a.nmb = (g.Mg + a.MB - 1) / a.MB;
  a.TW = 32 * g.sW;
  // rows: up to kTrSegs segments (row, w phase) per warp
  const int rows_max = (kTrSegs * kTrWarps) / g.sW;
  if (rows_max < 1) return p;  // sW > 32
  a.TH = g.OH < rows_max ? g.OH : rows_max;
  a.TD = 1;
  if (a.TH == g.OH && g.OD > 1) {
    a.TD = rows_max / a.TH;
    if (a.TD > g.OD) a.TD = g.OD;
    if (a.TD < 1) a.TD = 1;
  }
  a.nTw = (g.OW + a.TW - 1) / a.TW;
  a.nTh = (g.OH + a.TH - 1) / a.TH;
  a.nTd = (g.OD + a.TD - 1) / a.TD;
  a.BW = (a.TW - 1 + (g.KW - 1) * g.dW) / g.sW + 2;
  a.BH = (a.TH - 1 + (g.KH - 1) * g.dH) / g.sH + 2;
  a.BD = (a.TD - 1 + (g.KD - 1) * g.dD) / g.sD + 2;
  a.fd_kv = make_fastdiv((uint32_t)a.KV);
  a.fd_bh = make_fastdiv((uint32_t)a.BH);
  a.fd_brows = make_fastdiv((uint32_t)(a.BD * a.BH));
  const size_t box = (size_t)a.BD * a.BH * a.BW;
  const size_t per_c = (box + (size_t)a.KV * a.MB) * sizeof(float);
  if (a.KV > kTrMaxTaps) return p;
  const size_t lists = (size_t)kTrWarps * kTrSegs * a.KV * sizeof(int2) + 32;
  if (per_c + lists > kTrSmemBudget) return p;
  a.CC = (int)((kTrSmemBudget - lists) / per_c);
  if (a.CC > g.Cg) a.CC = g.Cg;
  if (a.CC > 32) a.CC = 32;
  // the box and the weights (each 16-byte aligned), then the per-warp tap lists
  p.smem = (size_t)a.CC * per_c + lists;
  p.blocks = (long long)g.N * g.G * a.nmb * a.nTd * a.nTh * a.nTw;
  if (p.blocks > 0x7fffffffLL) return p;
  p.ok = true;
  return p;
}

template <typename T>
int launch_tr_t(const ConvGeom& g, const TrPlan& p, const ConvArgs& args, cudaStream_t s) {
#define FCONV_TR_LAUNCH(MBV)                                                                    \
  if (p.a.MB == MBV) {                                                                          \
    auto k = convt_kernel<T, MBV>;                                                              \
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,        \
                                         (int)p.smem);                                          \
    if (e != cudaSuccess) return (int)e;                                                        \
    return launch_pdl(k, dim3((unsigned)p.blocks), dim3(kTrThreads), p.smem, s, g, p.a,         \
                      (const T*)args.x, (const T*)args.w, (const T*)args.b, (const T*)args.z,  \
                      (T*)args.y);                                                              \
  }
  FCONV_TR_LAUNCH(1)
  FCONV_TR_LAUNCH(2)
  FCONV_TR_LAUNCH(4)
  FCONV_TR_LAUNCH(8)
  FCONV_TR_LAUNCH(16)
#undef FCONV_TR_LAUNCH
  return (int)cudaErrorInvalidValue;
}

}  // namespace

bool transposed_supported(const ConvGeom& g) { return tr_plan(g).ok; }

int launch_transposed(const ConvGeom& g, const ConvArgs& a, void* stream) {
  const TrPlan p = tr_plan(g);
  if (!p.ok) return (int)cudaErrorInvalidValue;
  if (g.dtype == FCONV_F16) return launch_tr_t<__half>(g, p, a, (cudaStream_t)stream);
  return launch_tr_t<float>(g, p, a, (cudaStream_t)stream);
}

}  // namespace fconv
