// Direct FusedConv on CUDA cores: every dtype, spatial rank (1-3), group, stride,
// dilation and padding. One thread per output element; fp32 accumulation over the
// (C/group) x kernel taps in the order ci, kz, ky, kx; then + B + Z, the activation
// and one rounding to T.
//
// This is the general route: the tensor-core and depthwise kernels cover the common
// shapes faster. The index map is the one the manifest's params_ncdhw3d block carries
// (stride, dilation and the begin pads padD/padH/padW = effectivePad*), with taps that
// fall outside X reading zero.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "epilogue.cuh"
#include "fconv_internal.h"
#include "ptx.cuh"

namespace fconv {

// First tap t with i0 + t*d >= 0, and one past the last tap with i0 + t*d < n (k taps).
__device__ __forceinline__ int tap_lo(int i0, int d) { return i0 >= 0 ? 0 : (-i0 + d - 1) / d; }
__device__ __forceinline__ int tap_hi(int i0, int d, int n, int k) {
  if (i0 >= n) return 0;
  const int h = (n - i0 + d - 1) / d;
  return h < k ? h : k;
}

template <typename T>
__global__ void __launch_bounds__(256) direct_conv_kernel(ConvGeom g, const T* __restrict__ x,
                                                          const T* __restrict__ w,
                                                          const T* __restrict__ b,
                                                          const T* __restrict__ z,
                                                          T* __restrict__ y, long long total,
                                                          int w_in_smem) {
  extern __shared__ float wsm[];  // W widened to f32, when it fits
  ptx::pdl_wait();
  ptx::pdl_trigger();
  if (w_in_smem) {
    const int wcount = g.M * g.Cg * g.KV;  // at most 8192 when staged
    for (int i = threadIdx.x; i < wcount; i += blockDim.x) wsm[i] = to_f32(w[i]);
    __syncthreads();
  }
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    long long o;
    int m, n, ow, oh, od;
    if (total < 0x7fffffffLL) {  // 32-bit index decoding (the common case)
      const uint32_t i32 = (uint32_t)idx, P32 = (uint32_t)g.P;
      const uint32_t nm = i32 / P32, o32 = i32 - nm * P32;
      m = (int)(nm % (uint32_t)g.M);
      n = (int)(nm / (uint32_t)g.M);
      const uint32_t t = o32 / (uint32_t)g.OW;
      ow = (int)(o32 - t * (uint32_t)g.OW);
      oh = (int)(t % (uint32_t)g.OH);
      od = (int)(t / (uint32_t)g.OH);
      o = o32;
    } else {
      o = idx % g.P;
      const long long nm = idx / g.P;
      m = (int)(nm % g.M);
      n = (int)(nm / g.M);
      ow = (int)(o % g.OW);
      oh = (int)((o / g.OW) % g.OH);
      od = (int)(o / ((long long)g.OW * g.OH));
    }
    (void)o;
    const int grp = m / g.Mg;
    const int iz0 = od * g.sD - g.pD, iy0 = oh * g.sH - g.pH, ix0 = ow * g.sW - g.pW;
    // the taps that land inside X, per axis (no test in the inner loops)
    const int z0 = tap_lo(iz0, g.dD), z1 = tap_hi(iz0, g.dD, g.ID, g.KD);
    const int y0 = tap_lo(iy0, g.dH), y1 = tap_hi(iy0, g.dH, g.IH, g.KH);
    const int x0 = tap_lo(ix0, g.dW), x1 = tap_hi(ix0, g.dW, g.IW, g.KW);
    float acc = 0.0f;
    for (int ci = 0; ci < g.Cg; ++ci) {
      const T* xp = x + ((long long)n * g.C + (long long)grp * g.Cg + ci) * g.IS;
      const long long woff = ((long long)m * g.Cg + ci) * g.KV;
      for (int kz = z0; kz < z1; ++kz) {
        const int iz = iz0 + kz * g.dD;
        for (int ky = y0; ky < y1; ++ky) {
          const int iy = iy0 + ky * g.dH;
          const T* xrow = xp + ((long long)iz * g.IH + iy) * g.IW + ix0;
          const long long wr = woff + (kz * g.KH + ky) * g.KW;
          if (w_in_smem) {
            const float* wrow = wsm + wr;
#pragma unroll 4
            for (int kx = x0; kx < x1; ++kx) acc = fmaf(to_f32(xrow[kx * g.dW]), wrow[kx], acc);
          } else {
            const T* wrow = w + wr;
#pragma unroll 4
            for (int kx = x0; kx < x1; ++kx) acc = fmaf(to_f32(xrow[kx * g.dW]), to_f32(wrow[kx]), acc);
          }
        }
      }
    }
    float v = acc;
    if (b) v += to_f32(b[m]);
    if (z) v += to_f32(z[idx]);
    y[idx] = from_f32<T>(apply_act(g.act, v, g.alpha, g.beta));
  }
}

int launch_direct(const ConvGeom& g, const ConvArgs& a, void* stream) {
  const long long total = (long long)g.N * g.M * g.P;
  const int threads = 256;
  long long blocks = (total + threads - 1) / threads;
  if (blocks > 152LL * 64) blocks = 152LL * 64;
  if (blocks < 1) blocks = 1;
  cudaStream_t s = (cudaStream_t)stream;
  // W (all of it, widened to f32) is staged in shared memory when it takes at most 32 KB
  const long long wbytes = (long long)g.M * g.Cg * g.KV * 4;
  const int w_in_smem = wbytes <= 32 * 1024 ? 1 : 0;
  const size_t smem = w_in_smem ? (size_t)wbytes : 0;
  if (g.dtype == FCONV_F16)
    return launch_pdl(direct_conv_kernel<__half>, dim3((unsigned)blocks), dim3(threads), smem, s, g,
                      (const __half*)a.x, (const __half*)a.w, (const __half*)a.b,
                      (const __half*)a.z, (__half*)a.y, total, w_in_smem);
  return launch_pdl(direct_conv_kernel<float>, dim3((unsigned)blocks), dim3(threads), smem, s, g,
                    (const float*)a.x, (const float*)a.w, (const float*)a.b, (const float*)a.z,
                    (float*)a.y, total, w_in_smem);
}

}  // namespace fconv
