// fp32 FusedConv on the tcgen05 tensor cores with the 3xTF32 split (C/group a multiple of 32).
//
// Each f32 operand v is split into hi = v with its 13 low mantissa bits cleared (exactly a
// TF32 value) and lo = v - hi (exact in f32). The product of two operands is taken as
//   hi_a * hi_b + hi_a * lo_b + lo_a * hi_b
// three tcgen05.mma.kind::tf32 issues into one f32 accumulator; the dropped lo_a * lo_b term
// and the tensor core's TF32 reading of lo (its top 10 mantissa bits) leave a relative error
// near 2^-21 per product, well inside the fp32 tolerance, at tensor-core speed (the package's
// f32 subgroup-matrix variants have the same purpose: f32 convolutions on the matrix units).
//
// Layout as in the TMA-fed f16 kernel, with 32 f32 channels per 128-byte row: one prologue
// launch writes W's hi and lo copies in the K order (32-channel block, tap, channel) and X's
// hi and lo copies repacked as Xb[c/32][n][d][h][w][32]; for a chunk (block cb, tap t) each
// pixel box is one 5-D TMA box of a copy, TMA applying stride, dilation and zero padding.
// Warps of a persistent CTA: 8 epilogue (two sets of four, one per TMEM lane quarter), MMA,
// TMA producer. A stage holds W hi, W lo (16 KB each) and the X hi and lo boxes. The
// epilogue writes the raw f32 sums ([split][N][M][P]) and a reduce launch adds the splits in
// order and applies B, Z and the activation in f32 (accurate library functions), so every
// plan of this path has three launches: prologue, GEMM, reduce.
//
// Every mbarrier wait is bounded (2 s); a wait that gives up sets a shared abort flag and the
// device error word; the CTA waits for the MMAs and TMA loads it issued, frees TMEM and exits.
#include "tc_common.cuh"

#include <climits>
#include <cstring>

namespace fconv {
namespace {

constexpr int kF32Warps = 10;
constexpr int kF32Threads = kF32Warps * 32;
constexpr int kF32EpiWarps = 8;
constexpr int kF32MmaWarp = 8;
constexpr int kF32LoadWarp = 9;
constexpr int kBK32 = 32;                       // f32 K per chunk: one 128-byte row
constexpr uint32_t kW32Bytes = kMT * 128;       // one weights tile (hi or lo)

// Instruction descriptor of tcgen05.mma kind::tf32 with TF32 A and B (K-major) and an f32
// accumulator: D format (1 = f32) in [4,6), A/B formats (2 = TF32) in [7,10) and [10,13),
// N >> 3 in [17,23), M >> 4 in [24,29).
constexpr uint32_t idesc_tf32_f32(int M, int N) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_tf32(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

struct Tf32Args {
  BoxTiling t;
  float* part;
  int stages;
  int cbg;              // 32-channel blocks per group
  uint32_t px_bytes;    // bytes of one pixel box (rows * 128)
  uint32_t idesc;
};

struct Tf32Ctl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t acc_full[kMaxAcc];
  uint64_t acc_empty[kMaxAcc];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

template <int NPX>
__global__ void __launch_bounds__(kF32Threads, 1)
    igemm_tf32_kernel(const ConvGeom g, const Tf32Args a, const __grid_constant__ CUtensorMap tm_xhi,
                      const __grid_constant__ CUtensorMap tm_xlo,
                      const __grid_constant__ CUtensorMap tm_whi,
                      const __grid_constant__ CUtensorMap tm_wlo) {
  using AP = AccPlan<NPX, kF32EpiWarps>;
  constexpr uint32_t kStageBytes = 2 * kW32Bytes + 2 * NPX * 128;

  extern __shared__ uint8_t dsmem[];
  __shared__ Tf32Ctl ctl;

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
      ptx::mbar_init(ptx::smem_addr(&ctl.acc_empty[b]), kF32EpiWarps / AP::sets);
    }
    ptx::mbar_init(ptx::smem_addr(&ctl.drain), 1);
    ctl.abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kF32MmaWarp) {
    ptx::tmem_alloc(ptx::smem_addr(&ctl.tmem_base), AP::tmem_cols);
    ptx::tmem_relinquish();
  }
  if (warp == kF32LoadWarp && lane == 0) {
    ptx::prefetch_tmap(&tm_xhi);
    ptx::prefetch_tmap(&tm_xlo);
    ptx::prefetch_tmap(&tm_whi);
    ptx::prefetch_tmap(&tm_wlo);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  volatile int* abort_flag = &ctl.abort_flag;
  ptx::pdl_wait();  // the split copies come from the prologue launch
  const uint32_t tp = base + (uint32_t)S * kStageBytes + NPX * 16;

  if (warp == kF32LoadWarp) {
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
        int cb = un.c_begin / g.KV, tap = un.c_begin - (un.c_begin / g.KV) * g.KV;
        int kx = tap % g.KW, ky = (tap / g.KW) % g.KH, kz = tap / (g.KW * g.KH);
        for (int i = 0; i < un.nk; ++i) {
          if (!bounded_wait(ptx::smem_addr(&ctl.empty[st.idx]), st.phase ^ 1u, abort_flag)) {
            stop = true;
            break;
          }
          const uint32_t bar = ptx::smem_addr(&ctl.full[st.idx]);
          const uint32_t sbase = base + st.idx * kStageBytes;
          ptx::mbar_arrive_expect_tx(bar, 2 * kW32Bytes + 2 * a.px_bytes);
          const int kc = (un.c_begin + i) * kBK32;
          ptx::tma_load_2d(sbase, &tm_whi, kc, row0, bar);
          ptx::tma_load_2d(sbase + kW32Bytes, &tm_wlo, kc, row0, bar);
          const int cx = un.ow0 * g.sW - g.pW + kx * g.dW;
          const int cy = un.oh0 * g.sH - g.pH + ky * g.dH;
          const int cz = un.od0 * g.sD - g.pD + kz * g.dD;
          const int cn = (un.grp * a.cbg + cb) * g.N + un.n0;
          ptx::tma_load_5d(sbase + 2 * kW32Bytes, &tm_xhi, 0, cx, cy, cz, cn, bar);
          ptx::tma_load_5d(sbase + 2 * kW32Bytes + NPX * 128, &tm_xlo, 0, cx, cy, cz, cn, bar);
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
  } else if (warp == kF32MmaWarp) {
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
          const uint32_t whi = base + st.idx * kStageBytes;
          const uint32_t wlo = whi + kW32Bytes;
          const uint32_t xhi = whi + 2 * kW32Bytes;
          const uint32_t xlo = xhi + NPX * 128;
#pragma unroll
          for (int kk = 0; kk < kBK32 / 8; ++kk) {  // K = 8 TF32 (32 bytes) per MMA
            const uint32_t o = (uint32_t)kk * 32;
            mma_tf32(dacc, ptx::desc_sw128(whi + o), ptx::desc_sw128(xhi + o), a.idesc,
                     (i > 0 || kk > 0) ? 1u : 0u);
            mma_tf32(dacc, ptx::desc_sw128(whi + o), ptx::desc_sw128(xlo + o), a.idesc, 1u);
            mma_tf32(dacc, ptx::desc_sw128(wlo + o), ptx::desc_sw128(xhi + o), a.idesc, 1u);
          }
          ptx::mma_commit(ptx::smem_addr(&ctl.empty[st.idx]));
          st.next((uint32_t)S);
        }
        if (stop) break;
        ptx::mma_commit(ptx::smem_addr(&ctl.acc_full[acc.idx]));
        acc.next((uint32_t)AP::nacc);
      }
      ptx::mma_commit(ptx::smem_addr(&ctl.drain));
      drain_wait(ptx::smem_addr(&ctl.drain), 0);
    }
  } else {
    // ================================================================ epilogue (warps 0-7)
    box_epilogue<NPX, kActPartial, AP::nacc, AP::sets, AP::wpq>(
        g, a.t, nullptr, nullptr, nullptr, nullptr, a.part, ctl.acc_full, ctl.acc_empty,
        abort_flag, tmem, pix, tp + (uint32_t)warp * kTpBytes, warp, lane);
  }

  ptx::pdl_trigger();
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kF32MmaWarp) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, AP::tmem_cols);
  }
}

// ---------------------------------------------------------------- prologue
// hi = v with the 13 low mantissa bits cleared (a TF32 value), lo = v - hi (exact).
__device__ __forceinline__ void split_tf32(float v, float& hi, float& lo) {
  hi = __uint_as_float(__float_as_uint(v) & 0xFFFFE000u);
  lo = v - hi;
}

struct Tf32PrologueArgs {
  const float* w;
  float* whi;
  float* wlo;
  int wblocks;          // M: one block per output channel
  int Cg, KV;
  const float* x;
  float* xhi;
  float* xlo;
  int N, C;
  long long S;          // spatial positions of an image
  long long nx;         // blocks along the flattened positions (128 each)
};

// Blocks [0, M): W row m into the K order (32-channel block, tap, channel), split.
// Blocks M..: 32 channels x 128 flattened positions q = n*S + s of X, through a shared tile
// (loads coalesced along the positions, stores coalesced along the channels), split into
// Xb[c/32][q][32].
__global__ void __launch_bounds__(256) prologue_tf32_kernel(const Tf32PrologueArgs p) {
  __shared__ float tile[128][33];
  ptx::pdl_trigger();
  ptx::pdl_wait();
  long long b = blockIdx.x;
  if (b < p.wblocks) {
    const int m = (int)b;
    const int Kg = p.Cg * p.KV;
    const float* src = p.w + (long long)m * Kg;
    for (int k = threadIdx.x; k < Kg; k += blockDim.x) {
      const int cb = k / (32 * p.KV), rem = k - cb * 32 * p.KV;
      const int tap = rem >> 5, c = rem & 31;
      float hi, lo;
      split_tf32(src[(cb * 32 + c) * p.KV + tap], hi, lo);
      p.whi[(long long)m * Kg + k] = hi;
      p.wlo[(long long)m * Kg + k] = lo;
    }
    return;
  }
  b -= p.wblocks;
  const long long bx = b % p.nx;
  const int cb = (int)(b / p.nx);
  const long long NS = (long long)p.N * p.S;
  const long long q0 = bx * 128;
  // in: thread (channel half h, position j) loads 16 channels of position q0 + j
  {
    const int j = threadIdx.x & 127, h = threadIdx.x >> 7;
    const long long q = q0 + j;
    float v[16];
    if (q < NS) {
      const long long n = q / p.S, s = q - n * p.S;
      const float* xp = p.x + (n * p.C + (long long)cb * 32 + h * 16) * p.S + s;
#pragma unroll
      for (int c = 0; c < 16; ++c) v[c] = xp[(long long)c * p.S];
    } else {
#pragma unroll
      for (int c = 0; c < 16; ++c) v[c] = 0.0f;
    }
#pragma unroll
    for (int c = 0; c < 16; ++c) tile[j][h * 16 + c] = v[c];
  }
  __syncthreads();
  // out: warp w writes positions w, w + 8, ...; lane = channel (one 128-byte row each)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int j = warp; j < 128; j += 8) {
    const long long q = q0 + j;
    if (q >= NS) break;
    float hi, lo;
    split_tf32(tile[j][lane], hi, lo);
    const long long o = ((long long)cb * NS + q) * 32 + lane;
    p.xhi[o] = hi;
    p.xlo[o] = lo;
  }
}

// Y = act(sum_s partial[s] + B + Z) in f32, the splits added in order 0..S-1.
template <int ACT>
__global__ void __launch_bounds__(256) reduce_f32_kernel(const ConvGeom g, const float* part,
                                                         int splits, const float* b,
                                                         const float* z, float* y,
                                                         long long total) {
  ptx::pdl_wait();
  ptx::pdl_trigger();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    float acc = part[i];
    for (int s = 1; s < splits; ++s) acc += part[(long long)s * total + i];
    const int m = (int)((i / g.P) % g.M);
    if (b) acc += b[m];
    if (z) acc += z[i];
    y[i] = act_eval<ACT, false>(acc, g.alpha, g.beta);
  }
}

// ---------------------------------------------------------------- host side

struct Tf32Shape {
  bool ok;
  BoxShape box;
  int npx;
};

Tf32Shape tf32_shape(const ConvGeom& g, int max_px) {
  Tf32Shape t{};
  t.ok = g.dtype == FCONV_F32 && (g.Cg % kBK32) == 0 && g.sD <= 8 && g.sH <= 8 && g.sW <= 8 &&
         (long long)(g.C / 32) * g.N <= 0x7fffffffLL && (long long)g.N * g.IS < 0x7fffff00LL &&
         (long long)g.N * g.P * g.M < 0x7fffffffLL;
  if (!t.ok) return t;
  // a stage carries two copies of each operand: pixel tiles of at most 128
  t.npx = max_px >= 128 ? 128 : 64;
  t.box = box_shape(g, t.npx, 256 / g.sW, 256 / g.sH, 256 / g.sD);
  while (t.npx > 64 && t.box.rows <= t.npx / 2) t.npx /= 2;
  return t;
}

size_t rup(size_t v, size_t a) { return (v + a - 1) / a * a; }
size_t tf32_w_bytes(const ConvGeom& g) { return rup((size_t)g.M * g.Kg * 4, 1024); }
size_t tf32_x_bytes(const ConvGeom& g) { return rup((size_t)g.N * (size_t)g.IS * g.C * 4, 1024); }

template <int NPX>
int launch_tf32_t(const ConvGeom& g, const IgemmConfig& c, const Tf32Args& t, const CUtensorMap* m,
                  cudaStream_t s) {
  const size_t smem = (size_t)t.stages * (2 * kW32Bytes + 2 * NPX * 128) + 1024 +
                      (size_t)NPX * 16 + kF32EpiWarps * kTpBytes;
  cudaError_t e = cudaFuncSetAttribute(igemm_tf32_kernel<NPX>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int)e;
  return launch_pdl(igemm_tf32_kernel<NPX>, dim3((unsigned)c.grid), dim3(kF32Threads), smem, s, g,
                    t, m[0], m[1], m[2], m[3]);
}

}  // namespace

bool igemm_tf32_capable(const ConvGeom& g, int max_px) { return tf32_shape(g, max_px).ok; }

long long igemm_tf32_mtiles(const ConvGeom& g, int max_px) { return tf32_shape(g, max_px).box.boxes; }

int igemm_tf32_chunks(const ConvGeom& g) { return (g.Cg / kBK32) * g.KV; }

size_t igemm_tf32_workspace_bytes(const ConvGeom& g, const IgemmConfig& c) {
  return 2 * tf32_w_bytes(g) + 2 * tf32_x_bytes(g) +
         (size_t)c.split_k * (size_t)g.N * (size_t)g.M * (size_t)g.P * 4;
}

int launch_igemm_tf32(const ConvGeom& g, const IgemmConfig& c, const ConvArgs& a, void* stream) {
  cudaStream_t s = (cudaStream_t)stream;
  const Tf32Shape sh = tf32_shape(g, c.tile_n);
  if (!sh.ok) return (int)cudaErrorInvalidValue;
  EncodeTiledFn enc = tensor_map_encoder();
  if (!enc) return (int)cudaErrorNotSupported;
  uint8_t* ws = (uint8_t*)a.ws;
  const size_t wb = tf32_w_bytes(g), xb = tf32_x_bytes(g);
  float* whi = (float*)ws;
  float* wlo = (float*)(ws + wb);
  float* xhi = (float*)(ws + 2 * wb);
  float* xlo = (float*)(ws + 2 * wb + xb);
  float* part = (float*)(ws + 2 * wb + 2 * xb);
  {
    Tf32PrologueArgs pa{};
    pa.w = (const float*)a.w;
    pa.whi = whi;
    pa.wlo = wlo;
    pa.wblocks = g.M;
    pa.Cg = g.Cg;
    pa.KV = g.KV;
    pa.x = (const float*)a.x;
    pa.xhi = xhi;
    pa.xlo = xlo;
    pa.N = g.N;
    pa.C = g.C;
    pa.S = g.IS;
    pa.nx = ((long long)g.N * g.IS + 127) / 128;
    const long long blocks = (long long)g.M + pa.nx * (g.C / 32);
    if (blocks > 0x7fffffffLL) return (int)cudaErrorInvalidValue;
    const int e = launch_pdl(prologue_tf32_kernel, dim3((unsigned)blocks), dim3(256), 0, s, pa);
    if (e != 0) return e;
  }
  CUtensorMap maps[4];
  std::memset(maps, 0, sizeof(maps));
  const cuuint32_t e2[2] = {1, 1};
  for (int h = 0; h < 2; ++h) {
    const cuuint64_t dims[2] = {(cuuint64_t)g.Kg, (cuuint64_t)g.M};
    const cuuint64_t str[1] = {(cuuint64_t)g.Kg * 4};
    const cuuint32_t box[2] = {(cuuint32_t)kBK32, (cuuint32_t)kMT};
    if (enc(&maps[2 + h], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, h ? (void*)wlo : (void*)whi, dims, str,
            box, e2, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return (int)cudaErrorInvalidValue;
  }
  const BoxShape& bx = sh.box;
  const cuuint64_t cbn = (cuuint64_t)(g.C / 32) * (cuuint64_t)g.N;
  for (int h = 0; h < 2; ++h) {
    const cuuint64_t xdims[5] = {32, (cuuint64_t)g.IW, (cuuint64_t)g.IH, (cuuint64_t)g.ID, cbn};
    const cuuint64_t xstr[4] = {128, (cuuint64_t)g.IW * 128, (cuuint64_t)g.IH * g.IW * 128,
                                (cuuint64_t)g.ID * g.IH * g.IW * 128};
    const cuuint32_t xbox[5] = {32, (cuuint32_t)(bx.Wt * g.sW), (cuuint32_t)(bx.Ht * g.sH),
                                (cuuint32_t)(bx.Dt * g.sD), (cuuint32_t)bx.Nb};
    const cuuint32_t xes[5] = {1, (cuuint32_t)g.sW, (cuuint32_t)g.sH, (cuuint32_t)g.sD, 1};
    if (enc(&maps[h], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 5, h ? (void*)xlo : (void*)xhi, xdims, xstr,
            xbox, xes, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return (int)cudaErrorInvalidValue;
  }
  Tf32Args t{};
  t.t = make_box_tiling(g, bx, c.split_k, igemm_tf32_chunks(g), 1, sh.npx);
  t.part = part;
  t.stages = sh.npx == 128 ? 2 : 3;
  t.cbg = g.Cg / 32;
  t.px_bytes = (uint32_t)bx.rows * 128u;
  t.idesc = idesc_tf32_f32(kMT, (bx.rows + 15) / 16 * 16);
  int err = sh.npx == 128 ? launch_tf32_t<128>(g, c, t, maps, s) : launch_tf32_t<64>(g, c, t, maps, s);
  if (err != 0) return err;
  const long long total = (long long)g.N * g.M * g.P;
  long long blocks = (total + 255) / 256;
  if (blocks > 152LL * 32) blocks = 152LL * 32;
#define FCONV_RF32(ACT)                                                                         \
  err = launch_pdl(reduce_f32_kernel<ACT>, dim3((unsigned)blocks), dim3(256), 0, s, g,          \
                   (const float*)part, c.split_k, (const float*)a.b, (const float*)a.z,         \
                   (float*)a.y, total)
  FCONV_ACT_SWITCH(g.act, FCONV_RF32)
#undef FCONV_RF32
  return err;
}

int read_and_clear_tf32_error(void* stream, unsigned* value) {
  return read_and_clear_tc_error((cudaStream_t)stream, value);
}

}  // namespace fconv
