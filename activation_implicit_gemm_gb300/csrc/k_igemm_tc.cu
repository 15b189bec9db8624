// Implicit-GEMM FusedConv on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// GEMM view per group g (the package's implicit im2col routes, README variants
// implicit_im2col_tiled_reg / implicit_im2col_subgroup_matrix: "gathers logical im2col
// elements directly from X ... avoiding a materialized column scratch buffer"):
//   rows    = output pixels q = (n, od, oh, ow)            MMA M = 128 per tile
//   columns = output channels of the group (Mg)            MMA N = tile_n (16..256)
//   depth   = k = (ci, kz, ky, kx), Kg = C/group * prod(k) consumed 64 at a time
//   A[q, k] = X[n, g*Cg + ci, od*sD - pD + kz*dD, oh*sH - pH + ky*dH, ow*sW - pW + kx*dW]
//             (0 outside X),  B[m, k] = W[g*Mg + m, ci, kz, ky, kx]
//
// One CTA computes a 128 x tile_n output tile over a range of K chunks:
//   warps 0-3  gather A: thread t owns tile row t (one output pixel) and writes its 64
//              k values of the chunk as eight 16-byte pieces into the 128B-swizzled,
//              K-major shared-memory layout the MMA descriptor reads;
//   warp 5     loads B (weights, already K-major in OIDHW memory) the same way;
//   warp 4     allocates the TMEM accumulator (128 lanes x tile_n f32 columns), and one
//              lane issues tcgen05.mma (K = 16 per instruction) and tcgen05.commit;
//   warps 0-3  after the last chunk read the accumulator with tcgen05.ld (lane = pixel,
//              column = channel) and run the fused epilogue: + B[m] + Z, activation,
//              one rounding to f16, store to NCDHW Y.
// A shared-memory ring of `stages` chunks with full/empty mbarriers overlaps gather,
// weight loads and MMAs.
//
// Split-K (the package's implicit_im2col_tiled_reg_splitk variants: "partitions the ...
// reduction across workgroups when the unsplit output grid is too small, then combines
// raw partial sums and applies the bias and fused activation once"): with split_k > 1
// each CTA writes raw f32 partial sums to the workspace and splitk_reduce_kernel adds
// the splits in a fixed order (deterministic), then applies B, Z and the activation.
//
// Every mbarrier wait is bounded in time; a wait that gives up sets a shared abort flag
// and the device error word, and the CTA drains its MMAs, frees TMEM and exits.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "epilogue.cuh"
#include "fconv_internal.h"
#include "ptx.cuh"

namespace fconv {

__device__ unsigned g_device_error = 0;

namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kThreads = 192;
constexpr int kMaxStages = 8;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr unsigned kErrWaitTimeout = 1u;

struct TcArgs {
  const uint16_t* x;
  const uint16_t* w;
  const __half* b;
  const __half* z;
  __half* y;
  float* ws;           // split-K partials [split][N][M][P] (f32), or null
  int stages;
  int chunks;          // ceil(Kg / 64)
  int chunks_per_split;
  int ntiles;          // channel tiles per group
};

struct SharedCtl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t acc;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ bool bounded_wait(uint32_t bar, uint32_t parity,
                                             volatile int* abort_flag) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((i & 127u) == 0) {
      if (*abort_flag) return false;
      if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        atomicOr(&g_device_error, kErrWaitTimeout);
        return false;
      }
    }
  }
}

template <int BN>
__global__ void __launch_bounds__(kThreads, 1) igemm_tc_kernel(const ConvGeom g, const TcArgs a) {
  constexpr uint32_t kTmemCols = BN < 32 ? 32 : BN;
  constexpr uint32_t kABytes = kBM * kBK * 2;  // 16 KB
  constexpr uint32_t kBBytes = BN * kBK * 2;
  constexpr uint32_t kIdesc = ptx::idesc_f16_f32(kBM, BN);

  extern __shared__ uint8_t dsmem[];
  __shared__ SharedCtl ctl;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t raw = ptx::smem_addr(dsmem);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 1024-byte aligned operand ring
  const uint32_t stage_bytes = kABytes + kBBytes;

  const int grp = blockIdx.y / a.ntiles;
  const int ct = blockIdx.y - grp * a.ntiles;
  const int split = blockIdx.z;
  const int c_begin = split * a.chunks_per_split;
  const int c_end = min(c_begin + a.chunks_per_split, a.chunks);
  const int nchunks = c_end - c_begin;
  const int S = a.stages;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(ptx::smem_addr(&ctl.full[s]), 128 + 32);
      ptx::mbar_init(ptx::smem_addr(&ctl.empty[s]), 1);
    }
    ptx::mbar_init(ptx::smem_addr(&ctl.acc), 1);
    ctl.abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 4) {
    ptx::tmem_alloc(ptx::smem_addr(&ctl.tmem_base), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  volatile int* abort_flag = &ctl.abort_flag;

  const long long NP = (long long)g.N * g.P;

  if (warp < 4) {
    // ---------------------------------------------------------------- A gather
    const int r = tid;  // tile row
    const long long q = (long long)blockIdx.x * kBM + r;
    const bool row_ok = q < NP;
    int n = 0, od = 0, oh = 0, ow = 0;
    if (row_ok) {
      n = (int)(q / g.P);
      const long long o = q - (long long)n * g.P;
      ow = (int)(o % g.OW);
      oh = (int)((o / g.OW) % g.OH);
      od = (int)(o / ((long long)g.OW * g.OH));
    }
    const int iz0 = od * g.sD - g.pD, iy0 = oh * g.sH - g.pH, ix0 = ow * g.sW - g.pW;
    uint32_t mz = 0, my = 0, mx = 0;  // bit t: tap t along that axis lands inside X
    for (int t = 0; t < g.KD; ++t) { const int v = iz0 + t * g.dD; if (v >= 0 && v < g.ID) mz |= 1u << t; }
    for (int t = 0; t < g.KH; ++t) { const int v = iy0 + t * g.dH; if (v >= 0 && v < g.IH) my |= 1u << t; }
    for (int t = 0; t < g.KW; ++t) { const int v = ix0 + t * g.dW; if (v >= 0 && v < g.IW) mx |= 1u << t; }
    if (!row_ok) mz = 0;
    const uint16_t* xg = a.x + ((long long)n * g.C + (long long)grp * g.Cg) * g.IS;
    const int pix = (iz0 * g.IH + iy0) * g.IW + ix0;
    const int HW = g.IH * g.IW;
    const int step_y = g.dH * g.IW - g.KW * g.dW;       // toff change when kx wraps
    const int step_z = g.dD * HW - g.KH * g.dH * g.IW;  // toff change when ky wraps
    const uint32_t swz = (uint32_t)(r & 7);

    for (int i = 0; i < nchunks; ++i) {
      const int s = i % S;
      if (i >= S && !bounded_wait(ptx::smem_addr(&ctl.empty[s]), ((i / S) - 1) & 1, abort_flag))
        break;
      const int k0 = (c_begin + i) * kBK;
      int ci = k0 / g.KV;
      int tap = k0 - ci * g.KV;
      int kz = tap / (g.KH * g.KW);
      int rem = tap - kz * g.KH * g.KW;
      int ky = rem / g.KW;
      int kx = rem - ky * g.KW;
      int toff = kz * g.dD * HW + ky * g.dH * g.IW + kx * g.dW;
      const uint16_t* xc = xg + (long long)ci * g.IS + pix;
      int k = k0;
      const uint32_t arow = base + (uint32_t)s * stage_bytes + (uint32_t)r * 128u;
#pragma unroll 1
      for (int j = 0; j < 8; ++j) {
        uint32_t pk[4];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          uint32_t v = 0;
          if (k < g.Kg) {
            if ((mz >> kz) & (my >> ky) & (mx >> kx) & 1u) v = __ldg(xc + toff);
            ++k;
            ++kx;
            toff += g.dW;
            if (kx == g.KW) {
              kx = 0;
              ++ky;
              toff += step_y;
              if (ky == g.KH) {
                ky = 0;
                ++kz;
                toff += step_z;
                if (kz == g.KD) {
                  kz = 0;
                  toff = 0;
                  xc += g.IS;
                }
              }
            }
          }
          if (e & 1) pk[e >> 1] |= v << 16;
          else pk[e >> 1] = v;
        }
        ptx::st_shared_v4(arow + (((uint32_t)j ^ swz) << 4), pk[0], pk[1], pk[2], pk[3]);
      }
      ptx::fence_proxy_async_smem();
      ptx::mbar_arrive(ptx::smem_addr(&ctl.full[s]));
    }

    // ---------------------------------------------------------------- epilogue
    if (!*abort_flag && bounded_wait(ptx::smem_addr(&ctl.acc), 0, abort_flag)) {
      ptx::tc_fence_after();
      const long long obase = row_ok ? (long long)n * g.M * g.P + (q - (long long)n * g.P) : 0;
      const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 16) {
        float v[16];
        ptx::tmem_ld16(lane_addr + (uint32_t)c0, v);
        if (!row_ok) continue;
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          const int mc = ct * BN + c0 + jj;
          if (mc >= g.Mg) break;
          const int m = grp * g.Mg + mc;
          const long long yi = obase + (long long)m * g.P;
          if (a.ws) {
            a.ws[(long long)split * NP * g.M + yi] = v[jj];
          } else {
            float t = v[jj];
            if (a.b) t += __half2float(a.b[m]);
            if (a.z) t += __half2float(a.z[yi]);
            a.y[yi] = __float2half_rn(apply_act(g.act, t, g.alpha, g.beta));
          }
        }
      }
    }
  } else if (warp == 5) {
    // ---------------------------------------------------------------- B (weights)
    const bool vec = (g.Kg & 7) == 0;
    for (int i = 0; i < nchunks; ++i) {
      const int s = i % S;
      if (i >= S && !bounded_wait(ptx::smem_addr(&ctl.empty[s]), ((i / S) - 1) & 1, abort_flag))
        break;
      const int k0 = (c_begin + i) * kBK;
      const uint32_t bbase = base + (uint32_t)s * stage_bytes + kABytes;
      for (int p = lane; p < BN * 8; p += 32) {
        const int ml = p >> 3, j = p & 7;
        const int mc = ct * BN + ml;
        const int k = k0 + j * 8;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (mc < g.Mg && k < g.Kg) {
          const uint16_t* wp = a.w + (long long)(grp * g.Mg + mc) * g.Kg + k;
          if (vec) {
            v = ptx::ldg_nc_v4(wp);
          } else {
            uint32_t e[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) e[t] = (k + t < g.Kg) ? (uint32_t)__ldg(wp + t) : 0u;
            v = make_uint4(e[0] | (e[1] << 16), e[2] | (e[3] << 16), e[4] | (e[5] << 16),
                           e[6] | (e[7] << 16));
          }
        }
        ptx::st_shared_v4(bbase + (uint32_t)ml * 128u + ((uint32_t)(j ^ (ml & 7)) << 4), v.x, v.y,
                          v.z, v.w);
      }
      ptx::fence_proxy_async_smem();
      ptx::mbar_arrive(ptx::smem_addr(&ctl.full[s]));
    }
  } else if (warp == 4 && lane == 0) {
    // ---------------------------------------------------------------- MMA issue
    for (int i = 0; i < nchunks; ++i) {
      const int s = i % S;
      if (!bounded_wait(ptx::smem_addr(&ctl.full[s]), (i / S) & 1, abort_flag)) break;
      ptx::tc_fence_after();
      const uint32_t abase = base + (uint32_t)s * stage_bytes;
      const uint32_t bbase = abase + kABytes;
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk) {
        ptx::mma_f16(tmem, ptx::desc_sw128(abase + kk * 32), ptx::desc_sw128(bbase + kk * 32),
                     kIdesc, (i > 0 || kk > 0) ? 1u : 0u);
      }
      ptx::mma_commit(ptx::smem_addr(&ctl.empty[s]));
    }
    ptx::mma_commit(ptx::smem_addr(&ctl.acc));
    // do not free TMEM before every issued MMA has finished
    bounded_wait(ptx::smem_addr(&ctl.acc), 0, abort_flag);
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// Y = act(sum_s partial[s] + B + Z), the splits added in order 0..S-1.
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const ConvGeom g, const float* ws,
                                                            int splits, const __half* b,
                                                            const __half* z, __half* y,
                                                            long long total) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    float acc = ws[i];
    for (int s = 1; s < splits; ++s) acc += ws[(long long)s * total + i];
    const int m = (int)((i / g.P) % g.M);
    if (b) acc += __half2float(b[m]);
    if (z) acc += __half2float(z[i]);
    y[i] = __float2half_rn(apply_act(g.act, acc, g.alpha, g.beta));
  }
}

template <int BN>
int launch_bn(const ConvGeom& g, const IgemmConfig& c, const TcArgs& ta, cudaStream_t s) {
  const size_t smem = igemm_tc_smem_bytes(BN, c.stages);
  cudaError_t e = cudaFuncSetAttribute(igemm_tc_kernel<BN>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int)e;
  const long long rows = ((long long)g.N * g.P + kBM - 1) / kBM;
  dim3 grid((unsigned)rows, (unsigned)(g.G * ta.ntiles), (unsigned)c.split_k);
  igemm_tc_kernel<BN><<<grid, kThreads, smem, s>>>(g, ta);
  return (int)cudaGetLastError();
}

}  // namespace

int igemm_tc_stages(int tile_n) {
  if (tile_n >= 256) return 4;
  if (tile_n >= 128) return 6;
  return 4;
}

size_t igemm_tc_smem_bytes(int tile_n, int stages) {
  return (size_t)stages * (size_t)(kBM * kBK * 2 + tile_n * kBK * 2) + 1024;
}

size_t igemm_tc_workspace_bytes(const ConvGeom& g, const IgemmConfig& c) {
  if (c.split_k <= 1) return 0;
  return (size_t)c.split_k * (size_t)g.N * (size_t)g.M * (size_t)g.P * sizeof(float);
}

bool igemm_tc_supported(const ConvGeom& g) {
  if (g.dtype != FCONV_F16) return false;
  if (g.KD > 32 || g.KH > 32 || g.KW > 32) return false;
  // in-plane offsets, including those of padded taps, stay in 32-bit ints
  const long long span = (long long)(g.ID + g.pD + 1) * (g.IH + g.pH + 1) * (g.IW + g.pW + 1);
  if (span > INT_MAX / 2) return false;
  const long long rows = ((long long)g.N * g.P + kBM - 1) / kBM;
  if (rows > INT_MAX) return false;
  if ((long long)g.G * ((g.Mg + 15) / 16) > 65535) return false;
  return true;
}

int launch_igemm_tc(const ConvGeom& g, const IgemmConfig& c, const ConvArgs& a, void* stream) {
  cudaStream_t s = (cudaStream_t)stream;
  TcArgs ta;
  ta.x = (const uint16_t*)a.x;
  ta.w = (const uint16_t*)a.w;
  ta.b = (const __half*)a.b;
  ta.z = (const __half*)a.z;
  ta.y = (__half*)a.y;
  ta.ws = c.split_k > 1 ? (float*)a.ws : nullptr;
  ta.stages = c.stages;
  ta.chunks = (g.Kg + kBK - 1) / kBK;
  ta.chunks_per_split = (ta.chunks + c.split_k - 1) / c.split_k;
  ta.ntiles = (g.Mg + c.tile_n - 1) / c.tile_n;
  if (c.stages < 2 || c.stages > kMaxStages) return (int)cudaErrorInvalidValue;
  int err;
  switch (c.tile_n) {
    case 16: err = launch_bn<16>(g, c, ta, s); break;
    case 32: err = launch_bn<32>(g, c, ta, s); break;
    case 64: err = launch_bn<64>(g, c, ta, s); break;
    case 128: err = launch_bn<128>(g, c, ta, s); break;
    case 256: err = launch_bn<256>(g, c, ta, s); break;
    default: return (int)cudaErrorInvalidValue;
  }
  if (err != 0 || c.split_k <= 1) return err;
  const long long total = (long long)g.N * g.M * g.P;
  long long blocks = (total + 255) / 256;
  if (blocks > 152LL * 32) blocks = 152LL * 32;
  splitk_reduce_kernel<<<(unsigned)blocks, 256, 0, s>>>(g, (const float*)a.ws, c.split_k, ta.b,
                                                        ta.z, ta.y, total);
  return (int)cudaGetLastError();
}

int read_and_clear_device_error(void* stream, unsigned* value) {
  cudaStream_t s = (cudaStream_t)stream;
  unsigned v = 0;
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return (int)e;
  e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v));
  if (e != cudaSuccess) return (int)e;
  if (v) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero));
    if (e != cudaSuccess) return (int)e;
  }
  *value = v;
  return 0;
}

}  // namespace fconv
