// Grouped FusedConv with few channels per group on CUDA cores (the package's grouped
// large-kernel route, README variants conv2d-grouped-large-w4*: input windows shared across
// channels and columns, f32 accumulation), for every spatial rank, stride and dilation. The
// tensor cores do not pay here: a group's GEMM is a few channels wide and a few hundred deep,
// and the conv is bound by moving X, Z and Y.
//
// One CTA per (image n, group g, box of output pixels TD x TH x TW). The CTA stages
//   - the box's receptive field of the group's Cg input channels in shared memory, in X's own
//     precision: one 5-D TMA box (x start rounded down to a 16-byte multiple, positions
//     outside X filled with zeros, which is the convolution's zero padding), or, when X's rows
//     are not 16-byte multiples, rows copied by the warps with plain loads;
//   - the group's weights as f32 in the order [ci][tap][m] (while the TMA load is in flight),
//     so that the MG weights of one (ci, tap) are consecutive and read as broadcast 16-byte
//     vectors.
// Thread t computes output pixel t of the box for all MG output channels of the group: per
// (ci, tap) one shared-memory load of the input value, MG/4 vector loads of weights, MG FMAs.
// Then + B, + Z, the activation and one rounding to T; for each channel the box's pixels
// leave as consecutive elements of Y (coalesced across the warp). The wait for the TMA load
// is bounded in time; a wait that runs out sets the device error word and the CTA returns.
#include "tc_common.cuh"

#include <cstring>

namespace fconv {
namespace {

constexpr int kGrThreads = 256;
constexpr size_t kGrSmemBudget = 96 * 1024;

struct GroupedArgs {
  int TD, TH, TW;          // output box
  int BD, BH, BW;          // its input halo box (BW: staged width, 16-byte multiple)
  int nTd, nTh, nTw;       // boxes per axis
  int MG;                  // output channels per group computed by a thread (Mg rounded up to
                           // a power of two; the channels past Mg are computed from zero weights
                           // and not stored)
  int xalign;              // elements per 16 bytes (x starts are rounded down to a multiple)
  int tma;                 // halo box by TMA (1) or by plain loads (0)
  uint32_t box_bytes;      // bytes of the staged halo box
  uint32_t wfloats;        // floats of the staged weights (a multiple of 4)
};

template <typename T, int MG, int ACT>
__device__ __forceinline__ void grouped_body(const ConvGeom& g, const GroupedArgs& a, const T* __restrict__ x,
                                             const T* __restrict__ w, const T* __restrict__ b,
                                             const T* __restrict__ z, T* __restrict__ y,
                                             const CUtensorMap* tmap, const T* sx, float* sw,
                                             uint64_t* bar) {
  // the block: (n, g, box)
  long long blk = blockIdx.x;
  const int tw = (int)(blk % a.nTw); blk /= a.nTw;
  const int th = (int)(blk % a.nTh); blk /= a.nTh;
  const int td = (int)(blk % a.nTd); blk /= a.nTd;
  const int grp = (int)(blk % g.G);
  const int n = (int)(blk / g.G);
  const int od0 = td * a.TD, oh0 = th * a.TH, ow0 = tw * a.TW;
  const int iz0 = od0 * g.sD - g.pD, iy0 = oh0 * g.sH - g.pH, ix0 = ow0 * g.sW - g.pW;
  const int xs = ix0 >= 0 ? ix0 - ix0 % a.xalign : -((-ix0 + a.xalign - 1) / a.xalign) * a.xalign;
  const int bsz = a.BD * a.BH * a.BW;
  const uint32_t sbar = ptx::smem_addr(bar);
  if (a.tma) {
    if (threadIdx.x == 0) {
      ptx::mbar_arrive_expect_tx(sbar, a.box_bytes);
      ptx::tma_load_5d(ptx::smem_addr(sx), tmap, xs, iy0, iz0, grp * g.Cg, n, sbar);
    }
  } else {
    // rows of the halo box, one warp per row, four rows in flight
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rows = g.Cg * a.BD * a.BH;
    const T* xg = x + ((long long)n * g.C + (long long)grp * g.Cg) * g.IS;
    T* sxw = const_cast<T*>(sx);
    for (int r0 = warp * 4; r0 < rows; r0 += (kGrThreads / 32) * 4) {
      for (int bx = lane; bx < a.BW; bx += 32) {
        T v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int r = r0 + u;
          v[u] = from_f32<T>(0.0f);
          if (r < rows) {
            const int by = r % a.BH, bz = (r / a.BH) % a.BD, ci = r / (a.BH * a.BD);
            const int ix = xs + bx, iy = iy0 + by, iz = iz0 + bz;
            if (ix >= 0 && ix < g.IW && iy >= 0 && iy < g.IH && iz >= 0 && iz < g.ID)
              v[u] = xg[(long long)ci * g.IS + ((long long)iz * g.IH + iy) * g.IW + ix];
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (r0 + u < rows) sxw[(r0 + u) * a.BW + bx] = v[u];
      }
    }
  }
  // weights [ci][tap][m] (f32), zero for m >= Mg
  const T* wg = w + (long long)grp * g.Mg * g.Kg;
  for (int i = threadIdx.x; i < MG * g.Kg; i += blockDim.x) {
    const int m = i / g.Kg, k = i - m * g.Kg;  // W[m][k], k = ci * KV + tap
    sw[k * MG + m] = m < g.Mg ? to_f32(wg[i]) : 0.0f;
  }
  __syncthreads();
  if (a.tma) {
    volatile int never = 0;
    if (!bounded_wait(sbar, 0, &never)) {  // device error word set
      drain_wait(sbar, 0);                  // the load was issued: let it land first
      return;
    }
  }

  const int t = threadIdx.x;
  const int wt = t % a.TW, ht = (t / a.TW) % a.TH, dt = t / (a.TW * a.TH);
  const int od = od0 + dt, oh = oh0 + ht, ow = ow0 + wt;
  if (dt >= a.TD || od >= g.OD || oh >= g.OH || ow >= g.OW) return;
  float acc[MG];
#pragma unroll
  for (int m = 0; m < MG; ++m) acc[m] = 0.0f;
  const T* sxp = sx + ((dt * g.sD) * a.BH + ht * g.sH) * a.BW + (ix0 - xs) + wt * g.sW;
  const float4* swp = reinterpret_cast<const float4*>(sw);
  for (int ci = 0; ci < g.Cg; ++ci) {
    const T* sxc = sxp + ci * bsz;
    for (int kz = 0; kz < g.KD; ++kz) {
      for (int ky = 0; ky < g.KH; ++ky) {
        const T* row = sxc + (kz * g.dD * a.BH + ky * g.dH) * a.BW;
        const int k0 = ci * g.KV + (kz * g.KH + ky) * g.KW;
#pragma unroll 4
        for (int kx = 0; kx < g.KW; ++kx) {
          const float v = to_f32(row[kx * g.dW]);
          const int k = k0 + kx;
          if constexpr (MG % 4 == 0) {
#pragma unroll
            for (int q = 0; q < MG / 4; ++q) {
              const float4 wv = swp[k * (MG / 4) + q];
              acc[4 * q] = fmaf(v, wv.x, acc[4 * q]);
              acc[4 * q + 1] = fmaf(v, wv.y, acc[4 * q + 1]);
              acc[4 * q + 2] = fmaf(v, wv.z, acc[4 * q + 2]);
              acc[4 * q + 3] = fmaf(v, wv.w, acc[4 * q + 3]);
            }
          } else {
#pragma unroll
            for (int m = 0; m < MG; ++m) acc[m] = fmaf(v, sw[k * MG + m], acc[m]);
          }
        }
      }
    }
  }
  const long long pix = ((long long)od * g.OH + oh) * g.OW + ow;
#pragma unroll
  for (int m = 0; m < MG; ++m) {
    if (m >= g.Mg) break;
    const int mc = grp * g.Mg + m;
    const long long o = ((long long)n * g.M + mc) * g.P + pix;
    float v = acc[m];
    if (b) v += to_f32(b[mc]);
    if (z) v += to_f32(z[o]);
    y[o] = from_f32<T>(act_eval<ACT, sizeof(T) == 2>(v, g.alpha, g.beta));
  }
}

template <typename T, int MG>
__global__ void __launch_bounds__(kGrThreads) grouped_kernel(const ConvGeom g, const GroupedArgs a,
                                                             const T* __restrict__ x,
                                                             const T* __restrict__ w,
                                                             const T* __restrict__ b,
                                                             const T* __restrict__ z,
                                                             T* __restrict__ y,
                                                             const __grid_constant__ CUtensorMap tmap) {
  extern __shared__ __align__(1024) uint8_t gsm[];
  __shared__ uint64_t bar;
  T* sx = reinterpret_cast<T*>(gsm);                        // halo box (1024-byte aligned)
  float* sw = reinterpret_cast<float*>(gsm + ((a.box_bytes + 15u) & ~15u));
  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_addr(&bar), 1);
    ptx::fence_mbar_init();
    if (a.tma) ptx::prefetch_tmap(&tmap);
  }
  __syncthreads();
  ptx::pdl_wait();  // inputs may be the previous kernel's outputs
  ptx::pdl_trigger();
#define FCONV_GR_BODY(ACT) grouped_body<T, MG, ACT>(g, a, x, w, b, z, y, &tmap, sx, sw, &bar)
  FCONV_ACT_SWITCH(g.act, FCONV_GR_BODY)
#undef FCONV_GR_BODY
}

struct GroupedPlan {
  bool ok;
  GroupedArgs a;
  size_t smem;
  long long blocks;
};

int mg_instance(int Mg) {
  static const int inst[] = {1, 2, 4, 8, 16, 32};
  for (int v : inst)
    if (Mg <= v) return v;
  return 0;
}

GroupedPlan grouped_plan(const ConvGeom& g) {
  GroupedPlan p{};
  p.ok = false;
  if (mg_instance(g.Mg) == 0 || g.Cg > 16 || (long long)mg_instance(g.Mg) * g.Kg > 8192) return p;
  GroupedArgs& a = p.a;
  a.MG = mg_instance(g.Mg);
  const int es = g.dtype == FCONV_F16 ? 2 : 4;
  a.xalign = 16 / es;
  a.tma = (g.IW % a.xalign) == 0;
  a.wfloats = (uint32_t)((a.MG * g.Kg + 3) & ~3);
  // the largest box of at most 256 pixels whose halo box and weights fit the budget
  a.TW = g.OW < 64 ? g.OW : 64;
  for (;;) {
    a.TH = g.OH < kGrThreads / a.TW ? g.OH : kGrThreads / a.TW;
    if (a.TH < 1) a.TH = 1;
    a.TD = g.OD < kGrThreads / (a.TW * a.TH) ? g.OD : kGrThreads / (a.TW * a.TH);
    if (a.TD < 1) a.TD = 1;
    for (;;) {
      // staged width: the span of the box's taps plus the largest x alignment offset
      const int span = (a.TW - 1) * g.sW + (g.KW - 1) * g.dW + 1;
      a.BW = (span + a.xalign - 1 + a.xalign - 1) / a.xalign * a.xalign;
      a.BH = (a.TH - 1) * g.sH + (g.KH - 1) * g.dH + 1;
      a.BD = (a.TD - 1) * g.sD + (g.KD - 1) * g.dD + 1;
      a.box_bytes = (uint32_t)((size_t)g.Cg * a.BD * a.BH * a.BW * es);
      p.smem = (((size_t)a.box_bytes + 15) & ~(size_t)15) + (size_t)a.wfloats * 4;
      if (p.smem <= kGrSmemBudget) break;
      if (a.TD > 1) a.TD = (a.TD + 1) / 2;
      else if (a.TH > 1) a.TH = (a.TH + 1) / 2;
      else break;
    }
    if (p.smem <= kGrSmemBudget || a.TW == 1) break;
    a.TW = (a.TW + 1) / 2;
  }
  if (p.smem > kGrSmemBudget) return p;
  if (a.tma && (a.BW > 256 || a.BH > 256 || a.BD > 256 || g.Cg > 256)) a.tma = 0;
  a.nTd = (g.OD + a.TD - 1) / a.TD;
  a.nTh = (g.OH + a.TH - 1) / a.TH;
  a.nTw = (g.OW + a.TW - 1) / a.TW;
  p.blocks = (long long)g.N * g.G * a.nTd * a.nTh * a.nTw;
  if (p.blocks > 0x7fffffffLL) return p;
  p.ok = true;
  return p;
}

template <typename T>
int launch_grouped_t(const ConvGeom& g, const GroupedPlan& p, const ConvArgs& args, cudaStream_t s) {
  const T* x = (const T*)args.x;
  const T* w = (const T*)args.w;
  const T* b = (const T*)args.b;
  const T* z = (const T*)args.z;
  T* y = (T*)args.y;
  CUtensorMap tm;
  std::memset(&tm, 0, sizeof(tm));
  if (p.a.tma) {
    EncodeTiledFn enc = tensor_map_encoder();
    if (!enc) return (int)cudaErrorNotSupported;
    const cuuint64_t es = sizeof(T);
    const cuuint64_t dims[5] = {(cuuint64_t)g.IW, (cuuint64_t)g.IH, (cuuint64_t)g.ID,
                                (cuuint64_t)g.C, (cuuint64_t)g.N};
    const cuuint64_t str[4] = {(cuuint64_t)g.IW * es, (cuuint64_t)g.IH * g.IW * es,
                               (cuuint64_t)g.IS * es, (cuuint64_t)g.C * g.IS * es};
    const cuuint32_t box[5] = {(cuuint32_t)p.a.BW, (cuuint32_t)p.a.BH, (cuuint32_t)p.a.BD,
                               (cuuint32_t)g.Cg, 1};
    const cuuint32_t est[5] = {1, 1, 1, 1, 1};
    const CUresult cr = enc(&tm, sizeof(T) == 2 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                            5, (void*)x, dims, str, box, est, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS) return (int)cudaErrorInvalidValue;
  }
#define FCONV_GR_LAUNCH(MGV)                                                                   \
  if (p.a.MG == MGV) {                                                                         \
    auto k = grouped_kernel<T, MGV>;                                                           \
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,       \
                                         (int)p.smem);                                         \
    if (e != cudaSuccess) return (int)e;                                                       \
    return launch_pdl(k, dim3((unsigned)p.blocks), dim3(kGrThreads), p.smem, s, g, p.a, x, w, b, \
                      z, y, tm);                                                               \
  }
  FCONV_GR_LAUNCH(1)
  FCONV_GR_LAUNCH(2)
  FCONV_GR_LAUNCH(4)
  FCONV_GR_LAUNCH(8)
  FCONV_GR_LAUNCH(16)
  FCONV_GR_LAUNCH(32)
#undef FCONV_GR_LAUNCH
  return (int)cudaErrorInvalidValue;
}

}  // namespace

bool grouped_supported(const ConvGeom& g) { return grouped_plan(g).ok; }

int launch_grouped(const ConvGeom& g, const ConvArgs& a, void* stream) {
  const GroupedPlan p = grouped_plan(g);
  if (!p.ok) return (int)cudaErrorInvalidValue;
  if (g.dtype == FCONV_F16) return launch_grouped_t<__half>(g, p, a, (cudaStream_t)stream);
  return launch_grouped_t<float>(g, p, a, (cudaStream_t)stream);
}

int read_and_clear_grouped_error(void* stream, unsigned* value) {
  return read_and_clear_tc_error((cudaStream_t)stream, value);
}

}  // namespace fconv
