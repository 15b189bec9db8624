// Implicit-GEMM FusedConv on the 5th-generation tensor cores (tcgen05, sm_103a): the
// TMA-fed kernel for C/group a multiple of 64, the split-K reduction shared by both
// tensor-core kernels, and the host dispatch between the two ways the A operand reaches
// shared memory:
//   patch (k_igemm_patch.cu): each tile's NC(D)HW input patch arrives by TMA and builder
//     warps write the A rows from it; any C/group, no workspace
//   TMA-fed (this file): X is repacked into 64-channel blocks with channels innermost by a
//     prologue launch, Xb[c/64][n][d][h][w][64], and every A chunk is one 5-D TMA box of it
//
// TMA-fed kernel. A tile is a box of up to 256 output pixels and 128 output channels
// (tc_common.cuh, channel-major accumulator); for a chunk (64-channel block cb, tap t) the
// pixels' im2col rows are one 5-D TMA box of Xb at
// (0, ow0*sW - pW + kx*dW, oh0*sH - pH + ky*dH, od0*sD - pD + kz*dD, (g*Cg/64 + cb)*N + n0)
// with element strides (1, sW, sH, sD, 1): TMA applies stride, dilation and the zero
// padding, and writes the 128-byte-swizzled K-major rows the MMA reads. The weights come
// in the same (block, tap, channel) order from a copy the prologue writes, as 2-D boxes of
// 128 channels. No thread touches the operands. The repack exists because a TMA box of
// NC(D)HW X must start at an innermost (pixel) coordinate that is a multiple of 16 bytes,
// which a tap shift breaks; with 64 channels innermost the tap shift moves outer
// coordinates only.
//   warps 0-7  epilogue (two sets of four, one warp per TMEM lane quarter)
//   warp 8     TMEM allocation + MMA issue (tcgen05.mma.cta_group::1.kind::f16, M = 128
//              channels, N = the box's pixels rounded up to 16)
//   warp 9     TMA producer (weights and pixels of every chunk on one full barrier)
// A ring of `stages` chunks (weights 16 KB + pixels NPX*128 B each) with full/empty
// mbarriers; TMEM holds 512 / NPX accumulators so that epilogues overlap the MMAs.
//
// Split-K (README variants implicit_im2col_tiled_reg_splitk: the reduction is partitioned
// when the unsplit grid is too small, raw partial sums are combined, and the bias and
// activation are applied once): a work unit is (tile, split); units of a split plan write
// raw f32 partials to the workspace and splitk_reduce_kernel adds the splits in a fixed
// order, then applies B, Z and the activation (deterministic).
//
// Every mbarrier wait is bounded in time (2 s); a wait that gives up sets a shared abort
// flag and the device error word, and the CTA stops issuing work, waits (with a limit of
// its own, ignoring the flag) for the MMAs and TMA loads it already issued, frees TMEM and
// exits.
#include "tc_common.cuh"

#include <climits>
#include <cstring>
#include <mutex>

namespace fconv {
namespace {

constexpr int kTmaWarps = 10;
constexpr int kTmaThreads = kTmaWarps * 32;
constexpr int kTmaEpiWarps = 8;
constexpr int kTmaMmaWarp = 8;
constexpr int kTmaLoadWarp = 9;

// Shared-memory ring depth for a pixel tile: as many (weights 16 KB + pixels) chunks as fit
// in 180 KB (the rest holds the pixel table, the bias and the epilogue's transpose tiles),
// at most kMaxStages.
constexpr int stages_for(int npx) {
  const int st = (180 * 1024) / (kMT * kBK * 2 + npx * kBK * 2);
  const int capped = st > kMaxStages ? kMaxStages : st;
  return capped < 2 ? 2 : capped;
}

struct TmaArgs {
  BoxTiling t;
  const __half* b;
  const __half* z;
  __half* y;
  float* part;
  int stages;
  int cbg;              // 64-channel blocks per group
  uint32_t px_bytes;    // bytes of one pixel box (rows * 128)
  uint32_t idesc;       // MMA instruction descriptor (M = 128, N = pixels rounded to 16)
};

struct TmaCtl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t acc_full[kMaxAcc];
  uint64_t acc_empty[kMaxAcc];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

template <int NPX, bool SPLIT>
__global__ void __launch_bounds__(kTmaThreads, 1)
    igemm_tma_kernel(const ConvGeom g, const TmaArgs a, const __grid_constant__ CUtensorMap tmap_x,
                     const __grid_constant__ CUtensorMap tmap_w) {
  using AP = AccPlan<NPX, kTmaEpiWarps>;
  constexpr uint32_t kStageBytes = kWBytes + NPX * kBK * 2;

  extern __shared__ uint8_t dsmem[];
  __shared__ TmaCtl ctl;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t base = (ptx::smem_addr(dsmem) + 1023u) & ~1023u;
  uint8_t* gbase = dsmem + (base - ptx::smem_addr(dsmem));
  const int S = a.stages;
  int4* pix = reinterpret_cast<int4*>(gbase + (size_t)S * kStageBytes);

  build_pixel_table(g, a.t, pix, NPX);
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(ptx::smem_addr(&ctl.full[s]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl.empty[s]), 1);
    }
    for (int b = 0; b < AP::nacc; ++b) {
      ptx::mbar_init(ptx::smem_addr(&ctl.acc_full[b]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl.acc_empty[b]), kTmaEpiWarps / AP::sets);
    }
    ptx::mbar_init(ptx::smem_addr(&ctl.drain), 1);
    ctl.abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kTmaMmaWarp) {
    ptx::tmem_alloc(ptx::smem_addr(&ctl.tmem_base), AP::tmem_cols);
    ptx::tmem_relinquish();
  }
  if (warp == kTmaLoadWarp && lane == 0) {
    ptx::prefetch_tmap(&tmap_x);
    ptx::prefetch_tmap(&tmap_w);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  volatile int* abort_flag = &ctl.abort_flag;
  ptx::pdl_wait();  // the repacked X and the weight copy come from the prologue launch
  // bias widened to f32 beside the staging tiles (read by the epilogue warps only)
  float* bias_s = nullptr;
  if (a.b && g.M <= kMaxSmemBias) {
    bias_s = reinterpret_cast<float*>(gbase + (size_t)S * kStageBytes + NPX * 16);
    stage_bias(a.b, bias_s, g.M);
  }
  // the epilogue warps' transpose tiles follow the bias
  const uint32_t tp = base + (uint32_t)S * kStageBytes + NPX * 16 + kMaxSmemBias * 4;
  __syncthreads();

  if (warp == kTmaLoadWarp) {
    // ================================================================ TMA producer
    if (lane == 0) {
      Ring st{0, 0};
      uint32_t armed = 0;
      UnitIter it;
      it.init(a.t, blockIdx.x, gridDim.x);
      bool stop = false;
      for (; it.u < a.t.units && !stop; it.next(a.t)) {
        if (*abort_flag) break;
        const BoxUnit un = it.unit(a.t);
        const int row0 = un.grp * g.Mg + un.ct * kMT;
        // chunk = (64-channel block cb, tap): stepped without division
        int cb = un.c_begin / g.KV, tap = un.c_begin - (un.c_begin / g.KV) * g.KV;
        int kx = tap % g.KW, ky = (tap / g.KW) % g.KH, kz = tap / (g.KW * g.KH);
        for (int i = 0; i < un.nk; ++i) {
          if (!bounded_wait(ptx::smem_addr(&ctl.empty[st.idx]), st.phase ^ 1u, abort_flag)) {
            stop = true;
            break;
          }
          const uint32_t bar = ptx::smem_addr(&ctl.full[st.idx]);
          const uint32_t sbase = base + st.idx * kStageBytes;
          ptx::mbar_arrive_expect_tx(bar, kWBytes + a.px_bytes);
          ptx::tma_load_2d(sbase, &tmap_w, (un.c_begin + i) * kBK, row0, bar);
          ptx::tma_load_5d(sbase + kWBytes, &tmap_x, 0, un.ow0 * g.sW - g.pW + kx * g.dW,
                           un.oh0 * g.sH - g.pH + ky * g.dH, un.od0 * g.sD - g.pD + kz * g.dD,
                           (un.grp * a.cbg + cb) * g.N + un.n0, bar);
          ++armed;
          st.next((uint32_t)S);
          if (++kx == g.KW) {
            kx = 0;
            if (++ky == g.KH) {
              ky = 0;
              if (++kz == g.KD) {
                kz = 0;
                ++cb;
              }
            }
          }
        }
      }
      if (*abort_flag) drain_armed(ctl.full, armed, S);
    }
  } else if (warp == kTmaMmaWarp) {
    // ================================================================ MMA issue
    if (lane == 0) {
      Ring st{0, 0}, acc{0, 0};
      UnitIter it;
      it.init(a.t, blockIdx.x, gridDim.x);
      bool stop = false;
      for (; it.u < a.t.units && !stop; it.next(a.t)) {
        if (*abort_flag) break;
        const BoxUnit un = it.unit(a.t);
        if (!bounded_wait(ptx::smem_addr(&ctl.acc_empty[acc.idx]), acc.phase ^ 1u, abort_flag)) break;
        ptx::tc_fence_after();
        const uint32_t dacc = tmem + acc.idx * AP::cols;
        for (int i = 0; i < un.nk; ++i) {
          if (!bounded_wait(ptx::smem_addr(&ctl.full[st.idx]), st.phase, abort_flag)) {
            stop = true;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t wbase = base + st.idx * kStageBytes;
          const uint32_t pbase = wbase + kWBytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            ptx::mma_f16(dacc, ptx::desc_sw128(wbase + kk * 32), ptx::desc_sw128(pbase + kk * 32),
                         a.idesc, (i > 0 || kk > 0) ? 1u : 0u);
          }
          ptx::mma_commit(ptx::smem_addr(&ctl.empty[st.idx]));
          st.next((uint32_t)S);
        }
        if (stop) break;
        ptx::mma_commit(ptx::smem_addr(&ctl.acc_full[acc.idx]));
        acc.next((uint32_t)AP::nacc);
      }
      // every issued MMA must be complete before TMEM is freed
      ptx::mma_commit(ptx::smem_addr(&ctl.drain));
      drain_wait(ptx::smem_addr(&ctl.drain), 0);
    }
  } else {
    // ================================================================ epilogue (warps 0-7)
    // one loop per activation, chosen once: the group loop carries no dispatch
#define FCONV_EPI_LOOP(ACT)                                                                      \
  box_epilogue<NPX, ACT, AP::nacc, AP::sets, AP::wpq>(g, a.t, a.b, bias_s, a.z, a.y, a.part,     \
                                                     ctl.acc_full, ctl.acc_empty, abort_flag, tmem, \
                                                     pix, tp + (uint32_t)warp * kTpBytes, warp, lane)
    if constexpr (SPLIT) {
      FCONV_EPI_LOOP(kActPartial);
    } else {
      FCONV_ACT_SWITCH(g.act, FCONV_EPI_LOOP)
    }
#undef FCONV_EPI_LOOP
  }

  ptx::pdl_trigger();  // this CTA's work is done: the next kernel may start
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kTmaMmaWarp) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, AP::tmem_cols);
  }
}

// ---------------------------------------------------------------- prologue
// Everything the TMA-fed kernel reads in a layout of its own is written by ONE launch,
// prologue_kernel: its first `wblocks` blocks write the weight copy (one output channel
// each), the others repack X. Both parts only move data.

// X (N, C, spatial S) -> Xb[c/64][n][s][64]. Block (x, cb) moves 64 channels of the
// flattened positions q = n*S + s in [128x, 128x + 128), across image boundaries when S is
// small. In: four 16-byte loads per thread (8 positions of one channel), all in flight,
// each stored as one 16-byte chunk of a channel row of the shared tile; chunk k of channel
// c sits at k ^ ((c / 8) % 8). Out: a thread takes two adjacent positions and 8 channels
// (lanes: the 8 channel groups of 4 position pairs): eight 32-bit loads, byte permutes
// that pair up the channels, and one 16-byte store per position, so a warp writes whole
// 128-byte rows of Xb; the chunk swizzle puts the 8 channel groups of a load on distinct
// banks. Needs S % 8 == 0 (a load never straddles two images) and N*S < 2^31 (32-bit
// position decoding); otherwise pack_x_scalar is used.
constexpr int kPackPitch = 136;  // halves per channel row (272 bytes, 16-byte aligned)
constexpr size_t kPackSmem = 64 * kPackPitch * 2;

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

__device__ __forceinline__ void pack_x_block(const uint16_t* __restrict__ x, uint16_t* __restrict__ xb,
                                             int N, int C, long long S, long long bx, int cb,
                                             uint16_t* t) {
  const long long NS = (long long)N * S;
  const long long q0 = bx * 128;
  const int rows = (int)min(128LL, NS - q0);  // positions of this block (a multiple of 8)
  uint4 buf[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int v = threadIdx.x + 256 * i;
    const int c = v >> 4, pv = v & 15;
    buf[i] = make_uint4(0, 0, 0, 0);
    if (pv * 8 < rows) {
      const uint32_t q = (uint32_t)(q0 + pv * 8);
      const uint32_t n = q / (uint32_t)S, sp = q - n * (uint32_t)S;
      buf[i] = ptx::ldg_nc_v4(x + (((long long)n * C + (long long)cb * 64 + c) * S + sp));
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int v = threadIdx.x + 256 * i;
    const int c = v >> 4, pv = v & 15;
    *reinterpret_cast<uint4*>(t + c * kPackPitch + ((pv ^ ((c >> 3) & 7)) * 8)) = buf[i];
  }
  __syncthreads();
  uint16_t* dst = xb + ((long long)cb * NS + q0) * 64;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int item = threadIdx.x + 256 * i;
    const int part = item & 7, pp = item >> 3;  // channels 8*part.., positions 2pp, 2pp+1
    const int p = 2 * pp;
    if (p >= rows) continue;
    const int sw = (((p >> 3) ^ part) << 3) + (p & 7);  // swizzled place of position p
    uint32_t wv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      wv[j] = *reinterpret_cast<const uint32_t*>(t + (8 * part + j) * kPackPitch + sw);
    uint32_t lo[4], hi[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      lo[e] = prmt(wv[2 * e], wv[2 * e + 1], 0x5410u);  // channels 2e, 2e+1 at position p
      hi[e] = prmt(wv[2 * e], wv[2 * e + 1], 0x7632u);  // the same at position p + 1
    }
    *reinterpret_cast<uint4*>(dst + (long long)p * 64 + 8 * part) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    *reinterpret_cast<uint4*>(dst + (long long)(p + 1) * 64 + 8 * part) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
  }
}

// Scalar repack for S % 8 != 0: one thread per (position, 8 channels), block bi of nb.
__device__ __forceinline__ void pack_x_scalar(const uint16_t* __restrict__ x, uint16_t* __restrict__ xb,
                                              int N, int C, long long S, long long bi, long long nb) {
  const long long NS = (long long)N * S;
  const long long total = NS * (C / 8);
  for (long long i = bi * 256 + threadIdx.x; i < total; i += nb * 256) {
    const long long q = i % NS;
    const int c8 = (int)(i / NS);  // group of 8 channels
    const long long n = q / S, sp = q - n * S;
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const long long c = (long long)c8 * 8 + 2 * e;
      w[e] = (uint32_t)x[(n * C + c) * S + sp] | ((uint32_t)x[(n * C + c + 1) * S + sp] << 16);
    }
    const int cb = c8 / 8, part = c8 % 8;
    *reinterpret_cast<uint4*>(xb + ((long long)cb * NS + q) * 64 + part * 8) =
        make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Weights in the TMA-fed kernel's K order k' = (64-channel block, tap, channel): wp[m][k'].
// One block per output channel: the row is staged in shared memory (16-byte loads when
// rows are 16-byte aligned), then each thread writes 8 consecutive k' as one 16-byte store.
__device__ __forceinline__ void prep_weights_row(const uint16_t* __restrict__ w, uint16_t* __restrict__ wp,
                                                 int m, int Cg, int KV, uint16_t* row) {
  const int Kg = Cg * KV;
  const uint16_t* src = w + (long long)m * Kg;
  if ((Kg % 8) == 0) {
    for (int v = threadIdx.x; v < Kg / 8; v += blockDim.x)
      reinterpret_cast<uint4*>(row)[v] = reinterpret_cast<const uint4*>(src)[v];
  } else {
    for (int k = threadIdx.x; k < Kg; k += blockDim.x) row[k] = src[k];
  }
  __syncthreads();
  uint16_t* dst = wp + (long long)m * Kg;
  for (int v = threadIdx.x; v < Kg / 8; v += blockDim.x) {
    uint32_t e[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int k = v * 8 + j;
      const int cb = k / (64 * KV), rem = k - cb * 64 * KV;
      const int tap = rem >> 6;
      e[j] = (uint32_t)row[(cb * 64 + (rem & 63)) * KV + tap];
    }
    reinterpret_cast<uint4*>(dst)[v] =
        make_uint4(e[0] | (e[1] << 16), e[2] | (e[3] << 16), e[4] | (e[5] << 16), e[6] | (e[7] << 16));
  }
}

struct PrologueArgs {
  const uint16_t* w;
  uint16_t* wp;         // weight copy, or null (no weight blocks)
  int wblocks;          // = M when wp, else 0
  int Cg, KV;
  const uint16_t* x;
  uint16_t* xp;
  int scalar;           // pack_x_scalar instead of pack_x_block
  int N, C;
  long long S;
  long long nx;         // pack blocks along the position axis
};

__global__ void __launch_bounds__(256) prologue_kernel(const PrologueArgs p) {
  extern __shared__ __align__(16) uint16_t psm[];
  ptx::pdl_trigger();  // the main kernel may set itself up meanwhile
  ptx::pdl_wait();     // X and W may be the previous kernel's outputs
  long long b = blockIdx.x;
  if (b < p.wblocks) {
    prep_weights_row(p.w, p.wp, (int)b, p.Cg, p.KV, psm);
    return;
  }
  b -= p.wblocks;
  const long long bx = b % p.nx;
  const int by = (int)(b / p.nx);
  if (p.scalar) pack_x_scalar(p.x, p.xp, p.N, p.C, p.S, bx, p.nx);
  else pack_x_block(p.x, p.xp, p.N, p.C, p.S, bx, by, psm);
}

// Y = act(sum_s partial[s] + B + Z), the splits added in order 0..S-1.
template <int ACT>
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const ConvGeom g, const float* part,
                                                            int splits, const __half* b,
                                                            const __half* z, __half* y,
                                                            long long total) {
  ptx::pdl_wait();  // the partials are the previous kernel's output
  ptx::pdl_trigger();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    float acc = part[i];
    for (int s = 1; s < splits; ++s) acc += part[(long long)s * total + i];
    const int m = (int)((i / g.P) % g.M);
    if (b) acc += __half2float(b[m]);
    if (z) acc += __half2float(z[i]);
    y[i] = __float2half_rn(act_eval<ACT, true>(acc, g.alpha, g.beta));
  }
}

// ------------------------------------------------------------------- host side

// Pixel box of the TMA-fed kernel: the A box spans Wt*sW x Ht*sH x Dt*sD positions, each at
// most 256 (TMA box limit).
struct TmaShape {
  bool ok;
  BoxShape box;
  int npx;  // pixel tile of the kernel instantiation (64, 128, 256)
};

TmaShape tma_shape(const ConvGeom& g, int max_px = kMaxPx) {
  TmaShape t{};
  t.ok = g.dtype == FCONV_F16 && (g.Cg % kBK) == 0 && g.sD <= 8 && g.sH <= 8 && g.sW <= 8 &&
         (long long)(g.C / 64) * g.N <= 0x7fffffffLL &&  // the TMA box's last dim
         (long long)g.N * g.IS / 128 < 0x7fffffffLL &&   // pack grid
         (long long)g.N * g.P * g.M < 0x7fffffffLL &&      // 32-bit unit decoding
         (size_t)g.Kg * 2 <= 200 * 1024;                   // weight row staged in shared memory
  if (!t.ok) return t;
  t.npx = max_px >= 256 ? 256 : max_px >= 128 ? 128 : 64;
  t.box = box_shape(g, t.npx, 256 / g.sW, 256 / g.sH, 256 / g.sD);
  while (t.npx > 64 && t.box.rows <= t.npx / 2) t.npx /= 2;  // a smaller instantiation holds it
  return t;
}

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Weight copy in the block order (unless the kernel is 1x1: then W's order is that order).
size_t tma_prep_bytes(const ConvGeom& g) {
  return g.KV != 1 ? round_up((size_t)g.M * g.Kg * 2, 1024) : 0;
}
size_t tma_pack_bytes(const ConvGeom& g) {
  return round_up((size_t)g.N * (size_t)g.IS * (size_t)g.C * 2, 1024);
}

template <int NPX, bool SPLIT>
int launch_tma_t(const ConvGeom& g, const IgemmConfig& c, const TmaArgs& t, const CUtensorMap& tx,
                 const CUtensorMap& tw, cudaStream_t s) {
  const size_t smem = (size_t)t.stages * (size_t)(kMT * kBK * 2 + NPX * kBK * 2) + 1024 +
                      (size_t)NPX * 16 + (size_t)kMaxSmemBias * 4 + kTmaEpiWarps * kTpBytes;
  cudaError_t e = cudaFuncSetAttribute(igemm_tma_kernel<NPX, SPLIT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int)e;
  return launch_pdl(igemm_tma_kernel<NPX, SPLIT>, dim3((unsigned)c.grid), dim3(kTmaThreads), smem,
                    s, g, t, tx, tw);
}

int launch_tma_path(const ConvGeom& g, const IgemmConfig& c, const ConvArgs& a, cudaStream_t s) {
  const TmaShape sh = tma_shape(g, c.tile_n);
  if (!sh.ok) return (int)cudaErrorInvalidValue;
  EncodeTiledFn enc = tensor_map_encoder();
  if (!enc) return (int)cudaErrorNotSupported;
  uint8_t* ws = (uint8_t*)a.ws;
  const size_t pb = tma_prep_bytes(g);
  const size_t xb_bytes = tma_pack_bytes(g);
  uint16_t* xpack = (uint16_t*)(ws + pb);
  {
    // one prologue launch: the weight copy (when the GEMM's K order is not W's) and X
    // repacked into 64-channel blocks
    PrologueArgs pa{};
    pa.w = (const uint16_t*)a.w;
    pa.wp = pb ? (uint16_t*)ws : nullptr;
    pa.wblocks = pb ? g.M : 0;
    pa.Cg = g.Cg;
    pa.KV = g.KV;
    pa.x = (const uint16_t*)a.x;
    pa.xp = xpack;
    pa.N = g.N;
    pa.C = g.C;
    pa.S = g.IS;
    size_t smem = pb ? (size_t)g.Kg * 2 : 0;
    long long pack_blocks;
    const long long NS = (long long)g.N * g.IS;
    if (g.IS % 8 == 0 && NS < 0x7fffff00LL) {
      pa.scalar = 0;
      pa.nx = (NS + 127) / 128;
      pack_blocks = pa.nx * (g.C / 64);
      if (smem < kPackSmem) smem = kPackSmem;
    } else {
      pa.scalar = 1;
      long long blocks = (NS * (g.C / 8) + 255) / 256;
      if (blocks > 152LL * 32) blocks = 152LL * 32;
      pa.nx = blocks;
      pack_blocks = blocks;
    }
    if (smem > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(prologue_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return (int)e;
    }
    const long long blocks = pa.wblocks + pack_blocks;
    if (blocks > 0x7fffffffLL) return (int)cudaErrorInvalidValue;
    const int e = launch_pdl(prologue_kernel, dim3((unsigned)blocks), dim3(256), smem, s, pa);
    if (e != 0) return e;
  }
  const uint16_t* wmat = pb ? (const uint16_t*)ws : (const uint16_t*)a.w;
  CUtensorMap tm;
  std::memset(&tm, 0, sizeof(tm));
  cuuint64_t dims[2] = {(cuuint64_t)g.Kg, (cuuint64_t)g.M};
  cuuint64_t strides[1] = {(cuuint64_t)g.Kg * 2};
  cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)kMT};
  cuuint32_t estr[2] = {1, 1};
  CUresult cr = enc(&tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, (void*)wmat, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return (int)cudaErrorInvalidValue;

  float* part = c.split_k > 1 ? (float*)(ws + pb + xb_bytes) : nullptr;
  const BoxShape& bx = sh.box;
  CUtensorMap tx;
  std::memset(&tx, 0, sizeof(tx));
  const cuuint64_t cbn = (cuuint64_t)(g.C / 64) * (cuuint64_t)g.N;
  cuuint64_t xdims[5] = {64, (cuuint64_t)g.IW, (cuuint64_t)g.IH, (cuuint64_t)g.ID, cbn};
  cuuint64_t xstr[4] = {128, (cuuint64_t)g.IW * 128, (cuuint64_t)g.IH * g.IW * 128,
                        (cuuint64_t)g.ID * g.IH * g.IW * 128};
  cuuint32_t xbox[5] = {64, (cuuint32_t)(bx.Wt * g.sW), (cuuint32_t)(bx.Ht * g.sH),
                        (cuuint32_t)(bx.Dt * g.sD), (cuuint32_t)bx.Nb};
  cuuint32_t xes[5] = {1, (cuuint32_t)g.sW, (cuuint32_t)g.sH, (cuuint32_t)g.sD, 1};
  cr = enc(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 5, (void*)(ws + pb), xdims, xstr, xbox, xes,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return (int)cudaErrorInvalidValue;
  TmaArgs t{};
  t.t = make_box_tiling(g, bx, c.split_k, (g.Kg + kBK - 1) / kBK, 1, sh.npx);
  t.b = (const __half*)a.b;
  t.z = (const __half*)a.z;
  t.y = (__half*)a.y;
  t.part = part;
  t.stages = stages_for(sh.npx);
  t.cbg = g.Cg / 64;
  t.px_bytes = (uint32_t)bx.rows * 128u;
  t.idesc = ptx::idesc_f16_f32(kMT, (bx.rows + 15) / 16 * 16);
  int err;
  const bool sp = c.split_k > 1;
  switch (sh.npx) {
#define FCONV_TMA_NPX(NPX)                                                                     \
  case NPX:                                                                                    \
    err = sp ? launch_tma_t<NPX, true>(g, c, t, tx, tm, s) : launch_tma_t<NPX, false>(g, c, t, tx, tm, s); \
    break;
    FCONV_TMA_NPX(64)
    FCONV_TMA_NPX(128)
    FCONV_TMA_NPX(256)
#undef FCONV_TMA_NPX
    default: return (int)cudaErrorInvalidValue;
  }
  if (err != 0 || !sp) return err;
  return launch_splitk_reduce(g, c.split_k, part, a.b, a.z, a.y, s);
}

}  // namespace

EncodeTiledFn tensor_map_encoder() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)p;
    else
      cudaGetLastError();
  });
  return fn;
}

int launch_splitk_reduce(const ConvGeom& g, int splits, const float* part, const void* b,
                         const void* z, void* y, void* stream) {
  const long long total = (long long)g.N * g.M * g.P;
  long long blocks = (total + 255) / 256;
  if (blocks > 152LL * 32) blocks = 152LL * 32;
  int err = 0;
#define FCONV_REDUCE(ACT)                                                                  \
  err = launch_pdl(splitk_reduce_kernel<ACT>, dim3((unsigned)blocks), dim3(256), 0, stream, g, part, \
                   splits, (const __half*)b, (const __half*)z, (__half*)y, total)
  FCONV_ACT_SWITCH(g.act, FCONV_REDUCE)
#undef FCONV_REDUCE
  return err;
}

bool igemm_tc_tma_capable(const ConvGeom& g) { return tma_shape(g).ok; }

bool igemm_tc_supported(const ConvGeom& g, int max_px) {
  if (g.dtype == FCONV_F32) return igemm_tf32_capable(g, max_px);
  return tma_shape(g, max_px).ok || igemm_patch_capable(g, max_px);
}

int igemm_tc_resolve_path(const ConvGeom& g, int max_px, int requested) {
  // fp32: the 3xTF32 kernel, fed by TMA boxes of the repacked copies
  if (g.dtype == FCONV_F32) return (requested != 1 && igemm_tf32_capable(g, max_px)) ? 2 : 0;
  if (requested == 2) return tma_shape(g, max_px).ok ? 2 : 0;
  if (requested == 1) return igemm_patch_capable(g, max_px) ? 1 : 0;
  if (tma_shape(g, max_px).ok) return 2;
  return igemm_patch_capable(g, max_px) ? 1 : 0;
}

size_t igemm_tc_workspace_bytes(const ConvGeom& g, const IgemmConfig& c) {
  if (g.dtype == FCONV_F32) return igemm_tf32_workspace_bytes(g, c);
  if (c.a_path == 1) return igemm_patch_workspace_bytes(g, c);
  size_t b = tma_prep_bytes(g) + tma_pack_bytes(g);
  if (c.split_k > 1) b += (size_t)c.split_k * (size_t)g.N * (size_t)g.M * (size_t)g.P * 4;
  return b;
}

int igemm_tc_launches(const ConvGeom& g, const IgemmConfig& c) {
  if (g.dtype == FCONV_F32) return 3;  // prologue, 3xTF32 GEMM, reduce + epilogue
  if (c.a_path == 1) return igemm_patch_launches(g, c);
  return 2 + (c.split_k > 1 ? 1 : 0);  // prologue, main kernel, split-K reduce
}

long long igemm_tc_mtiles(const ConvGeom& g, int a_path, int max_px) {
  if (g.dtype == FCONV_F32) return igemm_tf32_mtiles(g, max_px);
  if (a_path == 1) return igemm_patch_mtiles(g, max_px);
  return tma_shape(g, max_px).box.boxes;
}

int igemm_tc_chunks(const ConvGeom& g, int a_path, int tile_n) {
  if (g.dtype == FCONV_F32) return igemm_tf32_chunks(g);
  if (a_path == 1) return igemm_patch_chunks(g, tile_n);
  return (g.Kg + kBK - 1) / kBK;
}

int launch_igemm_tc(const ConvGeom& g, const IgemmConfig& c, const ConvArgs& a, void* stream) {
  if (g.dtype == FCONV_F32) return launch_igemm_tf32(g, c, a, stream);
  if (c.a_path == 1) return launch_igemm_patch(g, c, a, stream);
  return launch_tma_path(g, c, a, (cudaStream_t)stream);
}

int read_and_clear_device_error(void* stream, unsigned* value) {
  unsigned v1 = 0, v2 = 0, v3 = 0, v4 = 0, v5 = 0;
  int e = read_and_clear_tc_error((cudaStream_t)stream, &v1);
  if (e != 0) return e;
  e = read_and_clear_patch_error(stream, &v2);
  if (e != 0) return e;
  e = read_and_clear_grouped_error(stream, &v3);
  if (e != 0) return e;
  e = read_and_clear_dw_error(stream, &v4);
  if (e != 0) return e;
  e = read_and_clear_tf32_error(stream, &v5);
  if (e != 0) return e;
  *value = v1 | v2 | v3 | v4 | v5;
  return 0;
}

}  // namespace fconv
