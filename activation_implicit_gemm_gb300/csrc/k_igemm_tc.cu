// Implicit-GEMM FusedConv on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// GEMM view per group g (the package's implicit im2col routes, README variants
// implicit_im2col_tiled_reg / implicit_im2col_subgroup_matrix: im2col elements are
// gathered straight from X into the GEMM tiles, "avoiding a materialized column scratch
// buffer"):
//   rows    = output pixels q = (n, od, oh, ow)            MMA M = 128 per tile
//   columns = output channels of the group (Mg)            MMA N = BN (16..256)
//   depth   = k over (ci, tap), Kg = C/group * prod(kernel), consumed 64 per chunk
//   A[q, k] = X[n, g*Cg + ci, od*sD - pD + kz*dD, oh*sH - pH + ky*dH, ow*sW - pW + kx*dW]
//             (0 outside X),   B[m, k] = W[g*Mg + m, ci, kz, ky, kx]
// The K order is a free choice as long as A and B agree. With C/group a multiple of 8
// the kernel uses k = tap*Cg + ci ("channel-inner"): every 8-wide piece of a row is 8
// channels of one tap, so its validity is one test and its addresses one stride apart;
// with C/group a multiple of 64 it uses (64-channel block, tap, channel), so that all
// taps of a block reuse the same slab of X from L1.
// The weights are then read from a copy in that order (prep_weights_kernel, into the
// workspace); otherwise k = ci*KV + tap, W's own order.
//
// Persistent, warp-specialised CTA (one per SM), 14 warps:
//   warps 0-3   epilogue: tcgen05.ld of an accumulator (lane = pixel, column = channel),
//               + B[m] + Z, activation, one rounding to f16, NC(D)HW store;
//   warps 4-11  A gather, two sets of four warps taking alternate K chunks; thread t of a
//               set owns tile row t (one output pixel), loads its 64 k values of the chunk
//               (64 loads in flight) and writes them as eight 16-byte pieces into the
//               128-byte-swizzled K-major layout the MMA descriptor reads;
//   warp 12     allocates TMEM (two accumulators of BN f32 columns, so the epilogue of
//               one tile overlaps the main loop of the next) and one lane issues
//               tcgen05.mma (K = 16 each) and tcgen05.commit;
//   warp 13     one lane streams the weight tiles with TMA (zero fill past the edges).
// A ring of `stages` shared-memory chunks (A 16 KB + B BN*128 B each) with full/empty
// mbarriers connects gather/TMA -> MMA; acc_full/acc_empty connect MMA <-> epilogue.
//
// Split-K (README variants implicit_im2col_tiled_reg_splitk: the reduction is
// partitioned when the unsplit grid is too small, raw partial sums are combined, and
// the bias and activation are applied once): a work unit is (tile, split); units of a
// split plan write raw f32 partials to the workspace and splitk_reduce_kernel adds the
// splits in a fixed order, then applies B, Z and the activation (deterministic).
//
// Every mbarrier wait is bounded in time (2 s); a wait that gives up sets a shared abort
// flag and the device error word, and the CTA stops issuing work, drains its MMAs,
// frees TMEM and exits.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "epilogue.cuh"
#include "fastdiv.cuh"
#include "fconv_internal.h"
#include "ptx.cuh"

namespace fconv {

__device__ unsigned g_device_error = 0;

namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kWarps = 18;
constexpr int kThreads = kWarps * 32;
constexpr int kEpiWarp0 = 0;     // warps 0-7 (two per TMEM lane quarter)
constexpr int kEpiWarps = 8;
constexpr int kGatherWarp0 = 8;  // warps 8-15
constexpr int kMmaWarp = 16;
constexpr int kTmaWarp = 17;
constexpr int kMaxStages = 8;
constexpr int kMaxTab = 2048;    // tap (channel-inner) or k (generic) table entries
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr unsigned kErrWaitTimeout = 1u;

struct TcArgs {
  const uint16_t* x;
  const __half* b;
  const __half* z;
  __half* y;
  float* part;          // split-K partials [split][N][M][P] (f32), or null
  int stages;
  int chunks;           // ceil(Kg / 64)
  int chunks_per_split;
  int split;
  int ntiles;           // channel tiles per group
  long long row_tiles;  // ceil(N*P / 128)
  long long units;      // row_tiles * G * ntiles * split
  FastDiv fd_split, fd_gnt, fd_P, fd_OW, fd_OH;  // unit and pixel decoding
};

struct SharedCtl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ bool bounded_wait(uint32_t bar, uint32_t parity,
                                             volatile int* abort_flag) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (*abort_flag) return false;
      if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        atomicOr(&g_device_error, kErrWaitTimeout);
        return false;
      }
    }
  }
}

struct Unit {
  long long rt;   // row tile
  int grp, ct, sp;
  int c_begin, nk;
};

__device__ __forceinline__ Unit decode_unit(long long u, const TcArgs& a, int G) {
  Unit t;
  uint32_t r, sp, gct, rt;
  fast_divmod((uint32_t)u, a.fd_split, r, sp);
  fast_divmod(r, a.fd_gnt, rt, gct);
  t.sp = (int)sp;
  t.rt = rt;
  t.grp = (int)gct / a.ntiles;
  t.ct = (int)gct - t.grp * a.ntiles;
  t.c_begin = t.sp * a.chunks_per_split;
  t.nk = min(a.chunks_per_split, a.chunks - t.c_begin);
  return t;
}

// Bias, residual, activation and f16 rounding for the (up to) 16 channels of one pixel.
template <int ACT>
__device__ __forceinline__ void epi_store16(const float (&v)[16], const uint32_t (&zr)[16],
                                            const uint32_t (&br)[16], bool hz, bool hb,
                                            int nvalid, __half* yp, long long P, float alpha,
                                            float beta) {
  // all 16 results first (independent chains), then the stores
  __half h[16];
#pragma unroll
  for (int jj = 0; jj < 16; ++jj) {
    float t = v[jj];
    if (hb) t += __half2float(__ushort_as_half((unsigned short)br[jj]));
    if (hz) t += __half2float(__ushort_as_half((unsigned short)zr[jj]));
    h[jj] = __float2half_rn(act_eval<ACT, true>(t, alpha, beta));
  }
#pragma unroll
  for (int jj = 0; jj < 16; ++jj)
    if (jj < nvalid) yp[(long long)jj * P] = h[jj];
}

// As epi_store16, but the 16 results go to this lane's column of the warp's staging tile
// (channel-major, 64 bytes per channel row) for the vector store.
template <int ACT>
__device__ __forceinline__ void epi_stage16(const float (&v)[16], const uint32_t (&zr)[16],
                                            const uint32_t (&br)[16], bool hz, bool hb,
                                            uint32_t col, float alpha, float beta) {
  // all 16 results first (independent chains), then the shared-memory stores
  float o[16];
#pragma unroll
  for (int jj = 0; jj < 16; ++jj) {
    float t = v[jj];
    if (hb) t += __half2float(__ushort_as_half((unsigned short)br[jj]));
    if (hz) t += __half2float(__ushort_as_half((unsigned short)zr[jj]));
    o[jj] = act_eval<ACT, true>(t, alpha, beta);
  }
#pragma unroll
  for (int jj = 0; jj < 16; jj += 2) {
    // one packed conversion for two channels, then the two 2-byte stores
    const __half2 h2 = __floats2half2_rn(o[jj], o[jj + 1]);
    ptx::st_shared_u16(col + jj * 64, __half_as_ushort(__low2half(h2)));
    ptx::st_shared_u16(col + (jj + 1) * 64, __half_as_ushort(__high2half(h2)));
  }
}

template <int BN, bool CHAN>
__global__ void __launch_bounds__(kThreads, 1)
    igemm_tc_kernel(const ConvGeom g, const TcArgs a, const __grid_constant__ CUtensorMap tmap_w) {
  constexpr uint32_t kAccCols = BN < 32 ? 32 : BN;
  constexpr uint32_t kTmemCols = 2 * kAccCols;  // 64..512, a power of two
  constexpr uint32_t kABytes = kBM * kBK * 2;   // 16 KB
  constexpr uint32_t kBBytes = BN * kBK * 2;
  constexpr uint32_t kStageBytes = kABytes + kBBytes;
  constexpr uint32_t kIdesc = ptx::idesc_f16_f32(kBM, BN);

  extern __shared__ uint8_t dsmem[];
  __shared__ SharedCtl ctl;
  // channel-inner: per tap {offset in the X plane, kz | ky << 8 | kx << 16};
  // generic: per k {offset from the group's first channel plane, same tap bits}
  __shared__ __align__(16) int2 tab[kMaxTab];

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t base = (ptx::smem_addr(dsmem) + 1023u) & ~1023u;
  const int S = a.stages;
  const long long NP = (long long)g.N * g.P;
  const int HW = g.IH * g.IW;

  const int ntab = CHAN ? g.KV : g.Kg;
  for (int t = ntab + tid; t < ((ntab + 7) & ~7) && t < kMaxTab; t += kThreads) tab[t] = make_int2(0, 0);
  for (int t = tid; t < ntab && t < kMaxTab; t += kThreads) {
    const int ci = CHAN ? 0 : t / g.KV;
    const int tap = CHAN ? t : t - ci * g.KV;
    const int kx = tap % g.KW, ky = (tap / g.KW) % g.KH, kz = tap / (g.KW * g.KH);
    tab[t] = make_int2(ci * (int)g.IS + kz * g.dD * HW + ky * g.dH * g.IW + kx * g.dW,
                       kz | (ky << 8) | (kx << 16));
  }
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(ptx::smem_addr(&ctl.full[s]), 4 + 1);  // 4 gather warps + TMA
      ptx::mbar_init(ptx::smem_addr(&ctl.empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(ptx::smem_addr(&ctl.acc_full[b]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl.acc_empty[b]), kEpiWarps);
    }
    ptx::mbar_init(ptx::smem_addr(&ctl.drain), 1);
    ctl.abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(ptx::smem_addr(&ctl.tmem_base), kTmemCols);
    ptx::tmem_relinquish();
  }
  if (warp == kTmaWarp && lane == 0) ptx::prefetch_tmap(&tmap_w);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  volatile int* abort_flag = &ctl.abort_flag;

  if (warp >= kGatherWarp0 && warp < kGatherWarp0 + 8) {
    // ================================================================ A gather
    const int set = (warp - kGatherWarp0) >> 2;
    const int r = ((warp - kGatherWarp0) & 3) * 32 + lane;  // tile row
    const uint32_t swz = (uint32_t)(r & 7);
    uint32_t it = 0;
    for (long long u = blockIdx.x; u < a.units; u += gridDim.x) {
      if (*abort_flag) break;
      const Unit un = decode_unit(u, a, g.G);
      const long long q = un.rt * kBM + r;
      const bool row_ok = q < NP;
      int n = 0, od = 0, oh = 0, ow = 0;
      if (row_ok) {
        uint32_t nn, o, t1, w1, h1;
        fast_divmod((uint32_t)q, a.fd_P, nn, o);
        fast_divmod(o, a.fd_OW, t1, w1);
        fast_divmod(t1, a.fd_OH, o, h1);
        n = (int)nn; ow = (int)w1; oh = (int)h1; od = (int)o;
      }
      const int iz0 = od * g.sD - g.pD, iy0 = oh * g.sH - g.pH, ix0 = ow * g.sW - g.pW;
      uint32_t mz = 0, my = 0, mx = 0;  // bit t: tap t along that axis lands inside X
      for (int t = 0; t < g.KD; ++t) { const int v = iz0 + t * g.dD; if (v >= 0 && v < g.ID) mz |= 1u << t; }
      for (int t = 0; t < g.KH; ++t) { const int v = iy0 + t * g.dH; if (v >= 0 && v < g.IH) my |= 1u << t; }
      for (int t = 0; t < g.KW; ++t) { const int v = ix0 + t * g.dW; if (v >= 0 && v < g.IW) mx |= 1u << t; }
      if (!row_ok) mz = 0;
      const uint16_t* xg = a.x + ((long long)n * g.C + (long long)un.grp * g.Cg) * g.IS +
                           ((iz0 * g.IH + iy0) * g.IW + ix0);
      for (int i = 0; i < un.nk; ++i, ++it) {
        if ((int)(it & 1u) != set) continue;
        const int s = (int)(it % (uint32_t)S);
        if (it >= (uint32_t)S &&
            !bounded_wait(ptx::smem_addr(&ctl.empty[s]), ((it / S) - 1) & 1, abort_flag))
          break;
        const int k0 = (un.c_begin + i) * kBK;
        uint32_t v[64];
        if (CHAN && (g.Cg % kBK) == 0) {
          // K order (64-channel block, tap, channel): the chunk is 64 channels of one tap,
          // and the taps of a block follow each other, so the block's slab of X stays in
          // L1 across them. One validity test, 64 loads one channel plane apart, all in
          // flight before any store.
          const int chunk = un.c_begin + i;
          const int cb = chunk / g.KV;
          const int tap = chunk - cb * g.KV;
          const int ci = cb * kBK;
          const int2 ti = tab[tap];
          const bool ok = ((mz >> (ti.y & 0xff)) & (my >> ((ti.y >> 8) & 0xff)) & (mx >> (ti.y >> 16))) & 1u;
          if (ok) {
            const uint16_t* p = xg + (long long)ci * g.IS + ti.x;
#pragma unroll
            for (int e = 0; e < 64; ++e) v[e] = __ldg(p + (long long)e * g.IS);
          } else {
#pragma unroll
            for (int e = 0; e < 64; ++e) v[e] = 0u;
          }
        } else if (CHAN) {
          // eight pieces of 8 channels; each piece is one tap: one validity test, eight
          // loads one channel plane apart, all 64 loads in flight before any store
          int tap = k0 / g.Cg;
          int ci = k0 - tap * g.Cg;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int kk = k0 + 8 * j;
            uint32_t ok = 0;
            const uint16_t* p = xg;
            if (kk < g.Kg) {
              const int2 ti = tab[tap];
              ok = ((mz >> (ti.y & 0xff)) & (my >> ((ti.y >> 8) & 0xff)) & (mx >> (ti.y >> 16))) & 1u;
              p = xg + (long long)ci * g.IS + ti.x;
            }
            uint32_t(&v8)[8] = *reinterpret_cast<uint32_t(*)[8]>(&v[8 * j]);
            if (ok) {
              ptx::ld8_u16_nz(v8, p, g.IS * 2);
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e) v8[e] = 0u;
            }
            ci += 8;
            if (ci == g.Cg) { ci = 0; ++tap; }
          }
        } else {
          // per-k table: the table reads do not depend on each other or on the loads;
          // pieces of 8 past the end of K are skipped as a whole
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (k0 + 8 * j < g.Kg) {
              // the piece's 8 table entries first (broadcast reads, independent), then its
              // 8 loads back to back; the table is padded past Kg so the reads stay in it
              int2 te[8];
              const int4* tp = reinterpret_cast<const int4*>(&tab[k0 + 8 * j]);
#pragma unroll
              for (int h = 0; h < 4; ++h) {
                const int4 t4 = tp[h];
                te[2 * h] = make_int2(t4.x, t4.y);
                te[2 * h + 1] = make_int2(t4.z, t4.w);
              }
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const int2 ti = te[e];
                const uint32_t ok =
                    (k0 + 8 * j + e < g.Kg) &&
                    (((mz >> (ti.y & 0xff)) & (my >> ((ti.y >> 8) & 0xff)) & (mx >> (ti.y >> 16))) & 1u);
                v[8 * j + e] = ptx::ld1_u16(xg + ti.x, ok);
              }
            } else {
#pragma unroll
              for (int e = 8 * j; e < 8 * j + 8; ++e) v[e] = 0u;
            }
          }
        }
        const uint32_t arow = base + (uint32_t)s * kStageBytes + (uint32_t)r * 128u;
#pragma unroll
        for (int j = 0; j < 8; ++j) ptx::st_shared_pack8(arow + (((uint32_t)j ^ swz) << 4), &v[8 * j]);
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&ctl.full[s]));
      }
    }
  } else if (warp == kTmaWarp) {
    // ================================================================ weights by TMA
    if (lane == 0) {
      uint32_t it = 0;
      for (long long u = blockIdx.x; u < a.units; u += gridDim.x) {
        if (*abort_flag) break;
        const Unit un = decode_unit(u, a, g.G);
        const int row0 = un.grp * g.Mg + un.ct * BN;
        bool stop = false;
        for (int i = 0; i < un.nk; ++i, ++it) {
          const int s = (int)(it % (uint32_t)S);
          if (it >= (uint32_t)S &&
              !bounded_wait(ptx::smem_addr(&ctl.empty[s]), ((it / S) - 1) & 1, abort_flag)) {
            stop = true;
            break;
          }
          const uint32_t bar = ptx::smem_addr(&ctl.full[s]);
          ptx::mbar_arrive_expect_tx(bar, kBBytes);
          ptx::tma_load_2d(base + (uint32_t)s * kStageBytes + kABytes, &tmap_w,
                           (un.c_begin + i) * kBK, row0, bar);
        }
        if (stop) break;
      }
    }
  } else if (warp == kMmaWarp) {
    // ================================================================ MMA issue
    if (lane == 0) {
      uint32_t it = 0, tcount = 0;
      for (long long u = blockIdx.x; u < a.units; u += gridDim.x, ++tcount) {
        if (*abort_flag) break;
        const Unit un = decode_unit(u, a, g.G);
        const uint32_t b = tcount & 1u;
        if (tcount >= 2 &&
            !bounded_wait(ptx::smem_addr(&ctl.acc_empty[b]), ((tcount >> 1) - 1) & 1, abort_flag))
          break;
        ptx::tc_fence_after();
        const uint32_t dacc = tmem + b * kAccCols;
        bool stop = false;
        for (int i = 0; i < un.nk; ++i, ++it) {
          const int s = (int)(it % (uint32_t)S);
          if (!bounded_wait(ptx::smem_addr(&ctl.full[s]), (it / S) & 1, abort_flag)) {
            stop = true;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t abase = base + (uint32_t)s * kStageBytes;
          const uint32_t bbase = abase + kABytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            ptx::mma_f16(dacc, ptx::desc_sw128(abase + kk * 32), ptx::desc_sw128(bbase + kk * 32),
                         kIdesc, (i > 0 || kk > 0) ? 1u : 0u);
          }
          ptx::mma_commit(ptx::smem_addr(&ctl.empty[s]));
        }
        if (stop) break;
        ptx::mma_commit(ptx::smem_addr(&ctl.acc_full[b]));
      }
      // every issued MMA must be complete before TMEM is freed
      ptx::mma_commit(ptx::smem_addr(&ctl.drain));
      bounded_wait(ptx::smem_addr(&ctl.drain), 0, abort_flag);
    }
  } else {
    // ================================================================ epilogue (warps 0-7)
    const int q4 = (warp - kEpiWarp0) & 3;     // TMEM lane quarter
    const int half = (warp - kEpiWarp0) >> 2;  // which alternate 16-column groups
    const int r = q4 * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
    // 16-byte Y/Z vectors need 8-pixel groups inside one image (P % 8 == 0)
    const bool vec_io = (g.P % 8) == 0;
    const uint32_t yst = base + (uint32_t)S * kStageBytes + (uint32_t)(warp - kEpiWarp0) * 2048u;
    const uint32_t zst = yst + 1024u;
    uint32_t tcount = 0;
    for (long long u = blockIdx.x; u < a.units; u += gridDim.x, ++tcount) {
      if (*abort_flag) break;
      const Unit un = decode_unit(u, a, g.G);
      const uint32_t b = tcount & 1u;
      if (!bounded_wait(ptx::smem_addr(&ctl.acc_full[b]), (tcount >> 1) & 1, abort_flag)) break;
      ptx::tc_fence_after();
      const long long q = un.rt * kBM + r;
      const bool row_ok = q < NP;
      long long obase = 0;
      if (row_ok) {
        const long long n = fast_div((uint32_t)q, a.fd_P);
        obase = n * g.M * g.P + (q - n * g.P);
      }
      const int mc0 = un.ct * BN;
      // pixel group (8 consecutive pixels) this lane moves in the vector path
      const long long gq = un.rt * kBM + q4 * 32 + (lane & 3) * 8;
      const bool grp_ok = gq < NP;
      const long long gn = grp_ok ? (long long)fast_div((uint32_t)gq, a.fd_P) : 0;
      const long long gp = grp_ok ? gq - gn * g.P : 0;
#pragma unroll 1
      for (int c0 = half * 16; c0 < BN; c0 += 32) {
        float v[16];
        __syncwarp();
        ptx::tmem_ld16(lane_base + b * kAccCols + (uint32_t)c0, v);
        // the vector path needs every lane (shuffles, warp syncs); invalid rows there are
        // whole 8-pixel groups that are never stored
        if (!row_ok && !(vec_io && a.part == nullptr)) continue;
        const int mcb = mc0 + c0;
        const int nvalid = min(16, g.Mg - mcb);
        if (nvalid <= 0) continue;
        const long long yb = obase + (long long)(un.grp * g.Mg + mcb) * g.P;
        if (a.part) {
          float* pp = a.part + (long long)un.sp * NP * g.M + yb;
#pragma unroll
          for (int jj = 0; jj < 16; ++jj)
            if (jj < nvalid) pp[(long long)jj * g.P] = v[jj];
          continue;
        }
        const bool hz = a.z != nullptr, hb = a.b != nullptr;
        uint32_t zr[16], br[16];
        if (vec_io) {
          // Z and Y move as 16-byte vectors (8 pixels of one channel) through this warp's
          // staging tile [16 channels][32 pixels]; lane l owns pixel group l % 4 and
          // channels l / 4 and l / 4 + 8 for the vector moves
          const int m0 = un.grp * g.Mg + mcb;
          if (hz) {
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              const int ch = (lane >> 2) + 8 * t;
              uint4 zv = make_uint4(0, 0, 0, 0);
              if (grp_ok && ch < nvalid)
                zv = ptx::ldg_nc_v4(a.z + ((gn * g.M + m0 + ch) * g.P + gp));
              ptx::st_shared_v4(zst + ch * 64 + (lane & 3) * 16, zv.x, zv.y, zv.z, zv.w);
            }
            __syncwarp();
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) zr[jj] = ptx::ld_shared_u16(zst + jj * 64 + lane * 2);
          }
          if (hb) {
            const uint32_t bl = ptx::ld1_u16(a.b + m0 + (lane & 15), (lane & 15) < nvalid ? 1u : 0u);
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) br[jj] = __shfl_sync(0xffffffffu, bl, jj);
          }
#define FCONV_EPI16S(ACT) epi_stage16<ACT>(v, zr, br, hz, hb, yst + lane * 2, g.alpha, g.beta)
          FCONV_ACT_SWITCH(g.act, FCONV_EPI16S)
#undef FCONV_EPI16S
          __syncwarp();
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int ch = (lane >> 2) + 8 * t;
            if (grp_ok && ch < nvalid) {
              const uint4 yv = ptx::ld_shared_v4(yst + ch * 64 + (lane & 3) * 16);
              ptx::st_global_v4(a.y + ((gn * g.M + m0 + ch) * g.P + gp), yv);
            }
          }
          __syncwarp();
          continue;
        }
        if (hz) {
#pragma unroll
          for (int jj = 0; jj < 16; ++jj)
            zr[jj] = ptx::ld1_u16(a.z + yb + (long long)jj * g.P, jj < nvalid ? 1u : 0u);
        }
        if (hb) {
          const __half* bp = a.b + un.grp * g.Mg + mcb;
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) br[jj] = ptx::ld1_u16(bp + jj, jj < nvalid ? 1u : 0u);
        }
        __half* yp = a.y + yb;
#define FCONV_EPI16(ACT) epi_store16<ACT>(v, zr, br, hz, hb, nvalid, yp, g.P, g.alpha, g.beta)
        FCONV_ACT_SWITCH(g.act, FCONV_EPI16)
#undef FCONV_EPI16
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&ctl.acc_empty[b]));
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}


// ============================================================================
// TMA-fed variant (C/group a multiple of 64). X is first repacked into blocks of 64
// channels, channels innermost: Xb[c/64][n][d][h][w][64] (pack_x_kernel). A tile of
// output pixels is a box (Nb images x Dt x Ht x Wt, at most 128 pixels); for a chunk
// (64-channel block cb, tap t) its A operand is one 5-D TMA box of Xb at
// (0, ow0*sW - pW + kx*dW, oh0*sH - pH + ky*dH, od0*sD - pD + kz*dD, (g*Cg/64 + cb)*N + n0)
// with element strides (1, sW, sH, sD, 1): TMA applies stride, dilation and the zero
// padding, and writes the 128-byte-swizzled K-major rows the MMA reads. The weights come
// in the same (block, tap, channel) order. No thread touches the operands.
//   warps 0-7  epilogue (two warps per TMEM lane quarter, alternate 16-column groups)
//   warp 8     TMEM allocation + MMA issue
//   warp 9     TMA producer (A and B of every chunk on one full barrier)
// ============================================================================
constexpr int kTmaWarps = 10;
constexpr int kTmaThreads = kTmaWarps * 32;
constexpr int kTmaEpiWarps = 8;
constexpr int kTmaMmaWarp = 8;
constexpr int kTmaLoadWarp = 9;

struct TmaArgs {
  const __half* b;
  const __half* z;
  __half* y;
  float* part;
  int stages;
  int chunks, chunks_per_split, split, ntiles, cbg;
  int Nb, Dt, Ht, Wt, nTd, nTh, nTw;
  int rows;            // Nb*Dt*Ht*Wt <= 128
  int vec;             // 8-row groups are 16-byte aligned, contiguous runs of Y
  uint32_t a_bytes;
  long long units;
  FastDiv fd_split, fd_gnt, fd_nTw, fd_nTh, fd_nTd;
};

struct TmaUnit {
  int n0, od0, oh0, ow0;
  int grp, ct, sp, c_begin, nk;
};

__device__ __forceinline__ TmaUnit decode_tma_unit(long long u, const TmaArgs& a, int G) {
  TmaUnit t;
  uint32_t r, sp, gct, rt, tw, th, td;
  fast_divmod((uint32_t)u, a.fd_split, r, sp);
  fast_divmod(r, a.fd_gnt, rt, gct);
  t.sp = (int)sp;
  t.grp = (int)gct / a.ntiles;
  t.ct = (int)gct - t.grp * a.ntiles;
  fast_divmod(rt, a.fd_nTw, rt, tw);
  fast_divmod(rt, a.fd_nTh, rt, th);
  fast_divmod(rt, a.fd_nTd, rt, td);
  t.n0 = (int)rt * a.Nb;
  t.od0 = td * a.Dt;
  t.oh0 = th * a.Ht;
  t.ow0 = tw * a.Wt;
  t.c_begin = t.sp * a.chunks_per_split;
  t.nk = min(a.chunks_per_split, a.chunks - t.c_begin);
  return t;
}

template <int BN>
__global__ void __launch_bounds__(kTmaThreads, 1)
    igemm_tma_kernel(const ConvGeom g, const TmaArgs a, const __grid_constant__ CUtensorMap tmap_x,
                     const __grid_constant__ CUtensorMap tmap_w) {
  constexpr uint32_t kAccCols = BN < 32 ? 32 : BN;
  constexpr uint32_t kTmemCols = 2 * kAccCols;
  constexpr uint32_t kABytes = kBM * kBK * 2;
  constexpr uint32_t kBBytes = BN * kBK * 2;
  constexpr uint32_t kStageBytes = kABytes + kBBytes;
  constexpr uint32_t kIdesc = ptx::idesc_f16_f32(kBM, BN);

  extern __shared__ uint8_t dsmem[];
  __shared__ SharedCtl ctl;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t base = (ptx::smem_addr(dsmem) + 1023u) & ~1023u;
  const int S = a.stages;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(ptx::smem_addr(&ctl.full[s]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl.empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(ptx::smem_addr(&ctl.acc_full[b]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl.acc_empty[b]), kTmaEpiWarps);
    }
    ptx::mbar_init(ptx::smem_addr(&ctl.drain), 1);
    ctl.abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kTmaMmaWarp) {
    ptx::tmem_alloc(ptx::smem_addr(&ctl.tmem_base), kTmemCols);
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

  if (warp == kTmaLoadWarp) {
    // ================================================================ TMA producer
    if (lane == 0) {
      uint32_t it = 0;
      for (long long u = blockIdx.x; u < a.units; u += gridDim.x) {
        if (*abort_flag) break;
        const TmaUnit un = decode_tma_unit(u, a, g.G);
        const int row0 = un.grp * g.Mg + un.ct * BN;
        bool stop = false;
        for (int i = 0; i < un.nk; ++i, ++it) {
          const int s = (int)(it % (uint32_t)S);
          if (it >= (uint32_t)S &&
              !bounded_wait(ptx::smem_addr(&ctl.empty[s]), ((it / S) - 1) & 1, abort_flag)) {
            stop = true;
            break;
          }
          const int chunk = un.c_begin + i;
          const int cb = chunk / g.KV;
          const int tap = chunk - cb * g.KV;
          const int kx = tap % g.KW, ky = (tap / g.KW) % g.KH, kz = tap / (g.KW * g.KH);
          const uint32_t bar = ptx::smem_addr(&ctl.full[s]);
          const uint32_t abase = base + (uint32_t)s * kStageBytes;
          ptx::mbar_arrive_expect_tx(bar, a.a_bytes + kBBytes);
          ptx::tma_load_5d(abase, &tmap_x, 0, un.ow0 * g.sW - g.pW + kx * g.dW,
                           un.oh0 * g.sH - g.pH + ky * g.dH, un.od0 * g.sD - g.pD + kz * g.dD,
                           (un.grp * a.cbg + cb) * g.N + un.n0, bar);
          ptx::tma_load_2d(abase + kABytes, &tmap_w, chunk * kBK, row0, bar);
        }
        if (stop) break;
      }
    }
  } else if (warp == kTmaMmaWarp) {
    // ================================================================ MMA issue
    if (lane == 0) {
      uint32_t it = 0, tcount = 0;
      for (long long u = blockIdx.x; u < a.units; u += gridDim.x, ++tcount) {
        if (*abort_flag) break;
        const TmaUnit un = decode_tma_unit(u, a, g.G);
        const uint32_t b = tcount & 1u;
        if (tcount >= 2 &&
            !bounded_wait(ptx::smem_addr(&ctl.acc_empty[b]), ((tcount >> 1) - 1) & 1, abort_flag))
          break;
        ptx::tc_fence_after();
        const uint32_t dacc = tmem + b * kAccCols;
        bool stop = false;
        for (int i = 0; i < un.nk; ++i, ++it) {
          const int s = (int)(it % (uint32_t)S);
          if (!bounded_wait(ptx::smem_addr(&ctl.full[s]), (it / S) & 1, abort_flag)) {
            stop = true;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t abase = base + (uint32_t)s * kStageBytes;
          const uint32_t bbase = abase + kABytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            ptx::mma_f16(dacc, ptx::desc_sw128(abase + kk * 32), ptx::desc_sw128(bbase + kk * 32),
                         kIdesc, (i > 0 || kk > 0) ? 1u : 0u);
          }
          ptx::mma_commit(ptx::smem_addr(&ctl.empty[s]));
        }
        if (stop) break;
        ptx::mma_commit(ptx::smem_addr(&ctl.acc_full[b]));
      }
      ptx::mma_commit(ptx::smem_addr(&ctl.drain));
      bounded_wait(ptx::smem_addr(&ctl.drain), 0, abort_flag);
    }
  } else {
    // ================================================================ epilogue (warps 0-7)
    const int q = warp & 3;      // TMEM lane quarter
    const int half = warp >> 2;  // which alternate 16-column groups
    const int r = q * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    const uint32_t yst = base + (uint32_t)S * kStageBytes + (uint32_t)warp * 2048u;
    const uint32_t zst = yst + 1024u;
    // this row's place in the pixel box
    const int wt = r % a.Wt;
    const int ht = (r / a.Wt) % a.Ht;
    const int dt = (r / (a.Wt * a.Ht)) % a.Dt;
    const int nb = r / (a.Wt * a.Ht * a.Dt);
    // the 8-row group this lane moves in the vector path
    const int gr = q * 32 + (lane & 3) * 8;
    const int gwt = gr % a.Wt, ght = (gr / a.Wt) % a.Ht, gdt = (gr / (a.Wt * a.Ht)) % a.Dt;
    const int gnb = gr / (a.Wt * a.Ht * a.Dt);
    const long long NP = (long long)g.N * g.P;
    uint32_t tcount = 0;
    for (long long u = blockIdx.x; u < a.units; u += gridDim.x, ++tcount) {
      if (*abort_flag) break;
      const TmaUnit un = decode_tma_unit(u, a, g.G);
      const uint32_t b = tcount & 1u;
      const int gn = un.n0 + gnb, god = un.od0 + gdt, goh = un.oh0 + ght, gow = un.ow0 + gwt;
      const bool grp_ok =
          gr < a.rows && gn < g.N && god < g.OD && goh < g.OH && gow < g.OW;
      const long long gpix = ((long long)god * g.OH + goh) * g.OW + gow;
      const int mc0 = un.ct * BN;
      // Z vectors of the next 16-column group, requested one group ahead (the first one
      // before waiting for the accumulator) so the load latency overlaps other work
      const bool zvec = a.vec && a.z != nullptr && a.part == nullptr;
      uint4 zn0 = make_uint4(0, 0, 0, 0), zn1 = make_uint4(0, 0, 0, 0);
      auto load_z = [&](int c0, uint4& z0, uint4& z1) {
        const int mcb = mc0 + c0;
        const long long zb = ((long long)gn * g.M + un.grp * g.Mg + mcb) * g.P + gpix;
        const int ch0 = lane >> 2, ch1 = (lane >> 2) + 8;
        z0 = (grp_ok && c0 < BN && mcb + ch0 < g.Mg) ? ptx::ldg_nc_v4(a.z + zb + (long long)ch0 * g.P)
                                                    : make_uint4(0, 0, 0, 0);
        z1 = (grp_ok && c0 < BN && mcb + ch1 < g.Mg) ? ptx::ldg_nc_v4(a.z + zb + (long long)ch1 * g.P)
                                                    : make_uint4(0, 0, 0, 0);
      };
      if (zvec) load_z(half * 16, zn0, zn1);
      if (!bounded_wait(ptx::smem_addr(&ctl.acc_full[b]), (tcount >> 1) & 1, abort_flag)) break;
      ptx::tc_fence_after();
      const int n = un.n0 + nb, od = un.od0 + dt, oh = un.oh0 + ht, ow = un.ow0 + wt;
      const bool row_ok = r < a.rows && n < g.N && od < g.OD && oh < g.OH && ow < g.OW;
      const long long obase =
          row_ok ? (long long)n * g.M * g.P + ((long long)od * g.OH + oh) * g.OW + ow : 0;
#pragma unroll 1
      for (int c0 = half * 16; c0 < BN; c0 += 32) {
        const uint4 zc0 = zn0, zc1 = zn1;
        if (zvec && c0 + 32 < BN) load_z(c0 + 32, zn0, zn1);
        float v[16];
        __syncwarp();
        ptx::tmem_ld16(lane_base + b * kAccCols + (uint32_t)c0, v);
        const int mcb = mc0 + c0;
        const int nvalid = min(16, g.Mg - mcb);
        if (nvalid <= 0) continue;
        const int m0 = un.grp * g.Mg + mcb;
        const bool hz = a.z != nullptr, hb = a.b != nullptr;
        uint32_t zr[16], br[16];
        if (a.part) {
          if (!row_ok) continue;
          float* pp = a.part + (long long)un.sp * NP * g.M + obase + (long long)m0 * g.P;
#pragma unroll
          for (int jj = 0; jj < 16; ++jj)
            if (jj < nvalid) pp[(long long)jj * g.P] = v[jj];
          continue;
        }
        if (a.vec) {
          if (hz) {
            ptx::st_shared_v4(zst + (lane >> 2) * 64 + (lane & 3) * 16, zc0.x, zc0.y, zc0.z, zc0.w);
            ptx::st_shared_v4(zst + ((lane >> 2) + 8) * 64 + (lane & 3) * 16, zc1.x, zc1.y, zc1.z,
                              zc1.w);
            __syncwarp();
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) zr[jj] = ptx::ld_shared_u16(zst + jj * 64 + lane * 2);
          }
          if (hb) {
            const uint32_t bl = ptx::ld1_u16(a.b + m0 + (lane & 15), (lane & 15) < nvalid ? 1u : 0u);
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) br[jj] = __shfl_sync(0xffffffffu, bl, jj);
          }
#define FCONV_EPI16S(ACT) epi_stage16<ACT>(v, zr, br, hz, hb, yst + lane * 2, g.alpha, g.beta)
          FCONV_ACT_SWITCH(g.act, FCONV_EPI16S)
#undef FCONV_EPI16S
          __syncwarp();
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int ch = (lane >> 2) + 8 * t;
            if (grp_ok && ch < nvalid) {
              const uint4 yv = ptx::ld_shared_v4(yst + ch * 64 + (lane & 3) * 16);
              ptx::st_global_v4(a.y + (((long long)gn * g.M + m0 + ch) * g.P + gpix), yv);
            }
          }
          __syncwarp();
          continue;
        }
        if (!row_ok) continue;
        const long long yb = obase + (long long)m0 * g.P;
        if (hz) {
#pragma unroll
          for (int jj = 0; jj < 16; ++jj)
            zr[jj] = ptx::ld1_u16(a.z + yb + (long long)jj * g.P, jj < nvalid ? 1u : 0u);
        }
        if (hb) {
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) br[jj] = ptx::ld1_u16(a.b + m0 + jj, jj < nvalid ? 1u : 0u);
        }
        __half* yp = a.y + yb;
#define FCONV_EPI16(ACT) epi_store16<ACT>(v, zr, br, hz, hb, nvalid, yp, g.P, g.alpha, g.beta)
        FCONV_ACT_SWITCH(g.act, FCONV_EPI16)
#undef FCONV_EPI16
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&ctl.acc_empty[b]));
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kTmaMmaWarp) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// X (N, C, spatial S) -> Xb[c/64][n][s][64]. Block (x, cb) moves 64 channels of the
// flattened positions q = n*S + s in [128x, 128x + 128): four 16-byte loads per thread
// (8 positions of one channel), all in flight, into a shared tile, then four 16-byte
// stores per thread (8 channels of one position). Needs S % 8 == 0 (a load never
// straddles two images); otherwise the scalar variant below is used.
__global__ void __launch_bounds__(256) pack_x_kernel(const uint16_t* __restrict__ x,
                                                     uint16_t* __restrict__ xb, int N, int C,
                                                     long long S) {
  constexpr int kPitch = 138;  // halves per channel row: 16-byte rows, few bank conflicts
  __shared__ __align__(16) uint16_t t[64 * kPitch];
  const long long NS = (long long)N * S;
  const long long q0 = (long long)blockIdx.x * 128;
  const int cb = blockIdx.y;
  uint4 buf[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int v = threadIdx.x + 256 * i;
    const int c = v >> 4, pv = v & 15;
    const long long q = q0 + pv * 8;
    buf[i] = make_uint4(0, 0, 0, 0);
    if (q < NS) {
      const long long n = q / S, sp = q - n * S;
      buf[i] = *reinterpret_cast<const uint4*>(x + ((n * C + (long long)cb * 64 + c) * S + sp));
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int v = threadIdx.x + 256 * i;
    const int c = v >> 4, pv = v & 15;
    uint32_t* d = reinterpret_cast<uint32_t*>(t + c * kPitch + pv * 8);  // 4-byte aligned
    d[0] = buf[i].x; d[1] = buf[i].y; d[2] = buf[i].z; d[3] = buf[i].w;
  }
  __syncthreads();
  uint16_t* dst = xb + ((long long)cb * NS + q0) * 64;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int o = threadIdx.x + 256 * i;
    const int p = o >> 3, part = o & 7;
    if (q0 + p >= NS) continue;
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      w[e] = (uint32_t)t[(8 * part + 2 * e) * kPitch + p] |
             ((uint32_t)t[(8 * part + 2 * e + 1) * kPitch + p] << 16);
    *reinterpret_cast<uint4*>(dst + (long long)p * 64 + 8 * part) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Scalar repack for S % 8 != 0: one thread per (position, 8 channels).
__global__ void __launch_bounds__(256) pack_x_scalar_kernel(const uint16_t* __restrict__ x,
                                                            uint16_t* __restrict__ xb, int N, int C,
                                                            long long S) {
  const long long NS = (long long)N * S;
  const long long total = NS * (C / 8);
  for (long long i = blockIdx.x * 256LL + threadIdx.x; i < total; i += (long long)gridDim.x * 256) {
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

// Weights in the GEMM's K order, zero padded to kpad columns: wp[m][k'] for k' < kpad.
// One block per output channel: the row is staged in shared memory (16-byte loads when
// rows are 16-byte aligned), then each thread writes 8 consecutive k' as one 16-byte
// store, reading the permuted sources from shared memory.
__device__ __forceinline__ int prep_src(int k, int Cg, int KV, int chan) {
  if (chan && (Cg % 64) == 0) {  // (64-channel block, tap, channel)
    const int cb = k / (64 * KV), rem = k - cb * 64 * KV;
    const int tap = rem >> 6;
    return (cb * 64 + (rem & 63)) * KV + tap;
  }
  if (chan) {  // (tap, channel)
    const int tap = k / Cg;
    return (k - tap * Cg) * KV + tap;
  }
  return k;
}

__global__ void __launch_bounds__(256) prep_weights_kernel(const uint16_t* __restrict__ w,
                                                           uint16_t* __restrict__ wp, int M,
                                                           int Cg, int KV, int kpad, int chan) {
  extern __shared__ uint16_t row[];
  const int m = blockIdx.x;
  const int Kg = Cg * KV;
  const uint16_t* src = w + (long long)m * Kg;
  if ((Kg % 8) == 0) {
    for (int v = threadIdx.x; v < Kg / 8; v += blockDim.x)
      reinterpret_cast<uint4*>(row)[v] = reinterpret_cast<const uint4*>(src)[v];
  } else {
    for (int k = threadIdx.x; k < Kg; k += blockDim.x) row[k] = src[k];
  }
  __syncthreads();
  uint16_t* dst = wp + (long long)m * kpad;
  for (int v = threadIdx.x; v < kpad / 8; v += blockDim.x) {
    uint32_t e[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int k = v * 8 + j;
      e[j] = k < Kg ? (uint32_t)row[prep_src(k, Cg, KV, chan)] : 0u;
    }
    reinterpret_cast<uint4*>(dst)[v] =
        make_uint4(e[0] | (e[1] << 16), e[2] | (e[3] << 16), e[4] | (e[5] << 16), e[6] | (e[7] << 16));
  }
}

// Y = act(sum_s partial[s] + B + Z), the splits added in order 0..S-1.
template <int ACT>
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const ConvGeom g, const float* part,
                                                            int splits, const __half* b,
                                                            const __half* z, __half* y,
                                                            long long total) {
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

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
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

bool channel_inner(const ConvGeom& g) { return (g.Cg % 8) == 0; }

// Pixel box of the TMA-fed kernel.
struct TmaShape {
  bool ok;
  int Nb, Dt, Ht, Wt, rows, vec;
  long long mtiles;
};

TmaShape tma_shape(const ConvGeom& g) {
  TmaShape t{};
  t.ok = (g.Cg % kBK) == 0 && g.sD <= 8 && g.sH <= 8 && g.sW <= 8 &&
         (long long)(g.C / 64) * g.N <= 0x7fffffffLL &&  // the TMA box's last dim
         (long long)g.N * g.IS / 128 < 0x7fffffffLL;     // pack grid
  if (!t.ok) return t;
  t.Wt = min(g.OW, min(128, 256 / g.sW));
  t.Ht = min(g.OH, min(128 / t.Wt, 256 / g.sH));
  t.Dt = min(g.OD, min(128 / (t.Wt * t.Ht), 256 / g.sD));
  const bool whole = t.Wt == g.OW && t.Ht == g.OH && t.Dt == g.OD;
  t.Nb = whole ? min(g.N, 128 / (t.Wt * t.Ht * t.Dt)) : 1;
  t.rows = t.Nb * t.Dt * t.Ht * t.Wt;
  t.mtiles = (long long)((g.N + t.Nb - 1) / t.Nb) * ((g.OD + t.Dt - 1) / t.Dt) *
             ((g.OH + t.Ht - 1) / t.Ht) * ((g.OW + t.Wt - 1) / t.Wt);
  t.vec = (g.P % 8 == 0) && ((t.Wt % 8 == 0 && g.OW % t.Wt == 0) || whole);
  // 8-pixel groups never straddle the 32-row lane quarters: rows is a multiple of 8 or
  // the groups past `rows` are simply invalid
  return t;
}

bool use_tma(const ConvGeom& g, int a_path) {
  if (a_path == 1) return false;
  return tma_shape(g).ok;
}

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

template <int BN, bool CHAN>
int launch_t(const ConvGeom& g, const IgemmConfig& c, const TcArgs& ta, const CUtensorMap& tm,
             cudaStream_t s) {
  const size_t smem = igemm_tc_smem_bytes(BN, c.stages);
  cudaError_t e = cudaFuncSetAttribute(igemm_tc_kernel<BN, CHAN>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int)e;
  igemm_tc_kernel<BN, CHAN><<<(unsigned)c.grid, kThreads, smem, s>>>(g, ta, tm);
  return (int)cudaGetLastError();
}

template <bool CHAN>
int launch_bn(const ConvGeom& g, const IgemmConfig& c, const TcArgs& ta, const CUtensorMap& tm,
              cudaStream_t s) {
  switch (c.tile_n) {
    case 16: return launch_t<16, CHAN>(g, c, ta, tm, s);
    case 32: return launch_t<32, CHAN>(g, c, ta, tm, s);
    case 64: return launch_t<64, CHAN>(g, c, ta, tm, s);
    case 128: return launch_t<128, CHAN>(g, c, ta, tm, s);
    case 256: return launch_t<256, CHAN>(g, c, ta, tm, s);
    default: return (int)cudaErrorInvalidValue;
  }
}

template <int BN>
int launch_tma_t(const ConvGeom& g, const IgemmConfig& c, const TmaArgs& t, const CUtensorMap& tx,
                 const CUtensorMap& tw, cudaStream_t s) {
  const size_t smem = (size_t)c.stages * (size_t)(kBM * kBK * 2 + BN * kBK * 2) + 1024 +
                      (size_t)kTmaEpiWarps * 2048;
  cudaError_t e = cudaFuncSetAttribute(igemm_tma_kernel<BN>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int)e;
  igemm_tma_kernel<BN><<<(unsigned)c.grid, kTmaThreads, smem, s>>>(g, t, tx, tw);
  return (int)cudaGetLastError();
}

int launch_reduce(const ConvGeom& g, const IgemmConfig& c, const float* part, const __half* b,
                  const __half* z, __half* y, cudaStream_t s) {
  const long long total = (long long)g.N * g.M * g.P;
  long long blocks = (total + 255) / 256;
  if (blocks > 152LL * 32) blocks = 152LL * 32;
#define FCONV_REDUCE(ACT)                                                                    \
  splitk_reduce_kernel<ACT><<<(unsigned)blocks, 256, 0, s>>>(g, part, c.split_k, b, z, y, total)
  FCONV_ACT_SWITCH(g.act, FCONV_REDUCE)
#undef FCONV_REDUCE
  return (int)cudaGetLastError();
}

}  // namespace

int igemm_tc_stages(int tile_n) {
  const int per = kBM * kBK * 2 + tile_n * kBK * 2;
  int st = (200 * 1024) / per;
  if (st > kMaxStages) st = kMaxStages;
  st &= ~1;  // the two gather sets alternate chunks: an even ring
  return st < 2 ? 2 : st;
}

size_t igemm_tc_smem_bytes(int tile_n, int stages) {
  // operand ring + 1 KB alignment slack + the epilogue warps' Y/Z staging tiles
  return (size_t)stages * (size_t)(kBM * kBK * 2 + tile_n * kBK * 2) + 1024 + 8 * 2048;
}

// Weight copy in GEMM order (when W itself cannot be read by TMA in that order).
static bool needs_prep(const ConvGeom& g) {
  if (channel_inner(g)) return !(g.KV == 1);  // 1x1: channel-inner order is W's order
  return (g.Kg % 8) != 0;                       // TMA rows must be 16-byte multiples
}

static size_t kpad_of(const ConvGeom& g) { return round_up((size_t)g.Kg, 8); }

static size_t prep_bytes(const ConvGeom& g) {
  return needs_prep(g) ? round_up((size_t)g.M * kpad_of(g) * 2, 1024) : 0;
}

static size_t pack_bytes(const ConvGeom& g, const IgemmConfig& c) {
  return use_tma(g, c.a_path) ? round_up((size_t)g.N * g.C * (size_t)g.IS * 2, 1024) : 0;
}

size_t igemm_tc_workspace_bytes(const ConvGeom& g, const IgemmConfig& c) {
  size_t b = prep_bytes(g) + pack_bytes(g, c);
  if (c.split_k > 1) b += (size_t)c.split_k * (size_t)g.N * (size_t)g.M * (size_t)g.P * 4;
  return b;
}

bool igemm_tc_tma_capable(const ConvGeom& g) { return tma_shape(g).ok; }

int igemm_tc_launches(const ConvGeom& g, const IgemmConfig& c) {
  return 1 + (needs_prep(g) ? 1 : 0) + (use_tma(g, c.a_path) ? 1 : 0) + (c.split_k > 1 ? 1 : 0);
}

long long igemm_tc_mtiles(const ConvGeom& g, int a_path) {
  if (use_tma(g, a_path)) return tma_shape(g).mtiles;
  return ((long long)g.N * g.P + kBM - 1) / kBM;
}

bool igemm_tc_supported(const ConvGeom& g) {
  if (g.dtype != FCONV_F16) return false;
  if (g.KD > 32 || g.KH > 32 || g.KW > 32) return false;
  if ((size_t)g.Kg * 2 > 200 * 1024) return false;  // weight row staged in shared memory
  // unit and pixel indices are decoded in 32 bits (every unit count is at most N*P*M)
  if ((long long)g.N * g.P * g.M >= 0x7fffffffLL) return false;
  if (channel_inner(g) ? g.KV > kMaxTab : g.Kg > kMaxTab) return false;
  // generic order: the per-k table holds ci * plane offsets in 32-bit ints
  if (!channel_inner(g) && (long long)g.Cg * g.IS > INT_MAX / 2) return false;
  // in-plane offsets, including those of padded taps, stay in 32-bit ints
  const long long span = (long long)(g.ID + g.pD + 1) * (g.IH + g.pH + 1) * (g.IW + g.pW + 1);
  if (span > INT_MAX / 2) return false;
  if ((long long)g.M * (long long)kpad_of(g) > INT_MAX) return false;
  return true;
}

int launch_igemm_tc(const ConvGeom& g, const IgemmConfig& c, const ConvArgs& a, void* stream) {
  cudaStream_t s = (cudaStream_t)stream;
  if (c.stages < 2 || c.stages > kMaxStages || (c.stages & 1)) return (int)cudaErrorInvalidValue;
  EncodeTiledFn enc = encode_fn();
  if (!enc) return (int)cudaErrorNotSupported;
  const bool chan = channel_inner(g);
  const uint16_t* wmat = (const uint16_t*)a.w;
  uint8_t* ws = (uint8_t*)a.ws;
  const size_t pb = prep_bytes(g);
  const int kpad = (int)kpad_of(g);
  if (pb) {
    uint16_t* wp = (uint16_t*)ws;
    const size_t rowbytes = (size_t)g.Kg * 2;
    if (rowbytes > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(prep_weights_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)rowbytes);
      if (e != cudaSuccess) return (int)e;
    }
    prep_weights_kernel<<<(unsigned)g.M, 256, rowbytes, s>>>((const uint16_t*)a.w, wp, g.M, g.Cg,
                                                             g.KV, kpad, chan ? 1 : 0);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return (int)e;
    wmat = wp;
  }
  const bool tma = use_tma(g, c.a_path);
  const size_t xb_bytes = pack_bytes(g, c);
  if (tma) {
    const long long S = g.IS;
    const long long NS = (long long)g.N * S;
    if (S % 8 == 0) {
      dim3 pg((unsigned)((NS + 127) / 128), (unsigned)(g.C / 64), 1);
      pack_x_kernel<<<pg, 256, 0, s>>>((const uint16_t*)a.x, (uint16_t*)(ws + pb), g.N, g.C, S);
    } else {
      long long blocks = (NS * (g.C / 8) + 255) / 256;
      if (blocks > 152LL * 32) blocks = 152LL * 32;
      pack_x_scalar_kernel<<<(unsigned)blocks, 256, 0, s>>>((const uint16_t*)a.x,
                                                             (uint16_t*)(ws + pb), g.N, g.C, S);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return (int)e;
  }
  const int wcols = pb ? kpad : g.Kg;
  CUtensorMap tm;
  std::memset(&tm, 0, sizeof(tm));
  cuuint64_t dims[2] = {(cuuint64_t)wcols, (cuuint64_t)g.M};
  cuuint64_t strides[1] = {(cuuint64_t)wcols * 2};
  cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)c.tile_n};
  cuuint32_t estr[2] = {1, 1};
  CUresult cr = enc(&tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, (void*)wmat, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return (int)cudaErrorInvalidValue;

  float* part = c.split_k > 1 ? (float*)(ws + pb + xb_bytes) : nullptr;
  if (tma) {
    const TmaShape sh = tma_shape(g);
    CUtensorMap tx;
    std::memset(&tx, 0, sizeof(tx));
    const cuuint64_t cbn = (cuuint64_t)(g.C / 64) * (cuuint64_t)g.N;
    cuuint64_t xdims[5] = {64, (cuuint64_t)g.IW, (cuuint64_t)g.IH, (cuuint64_t)g.ID, cbn};
    cuuint64_t xstr[4] = {128, (cuuint64_t)g.IW * 128, (cuuint64_t)g.IH * g.IW * 128,
                          (cuuint64_t)g.ID * g.IH * g.IW * 128};
    cuuint32_t xbox[5] = {64, (cuuint32_t)(sh.Wt * g.sW), (cuuint32_t)(sh.Ht * g.sH),
                          (cuuint32_t)(sh.Dt * g.sD), (cuuint32_t)sh.Nb};
    cuuint32_t xes[5] = {1, (cuuint32_t)g.sW, (cuuint32_t)g.sH, (cuuint32_t)g.sD, 1};
    cr = enc(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 5, (void*)(ws + pb), xdims, xstr, xbox, xes,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS) return (int)cudaErrorInvalidValue;
    TmaArgs t;
    t.b = (const __half*)a.b;
    t.z = (const __half*)a.z;
    t.y = (__half*)a.y;
    t.part = part;
    t.stages = c.stages;
    t.chunks = (g.Kg + kBK - 1) / kBK;
    t.chunks_per_split = (t.chunks + c.split_k - 1) / c.split_k;
    t.split = c.split_k;
    t.ntiles = (g.Mg + c.tile_n - 1) / c.tile_n;
    t.cbg = g.Cg / 64;
    t.Nb = sh.Nb; t.Dt = sh.Dt; t.Ht = sh.Ht; t.Wt = sh.Wt;
    t.nTd = (g.OD + sh.Dt - 1) / sh.Dt;
    t.nTh = (g.OH + sh.Ht - 1) / sh.Ht;
    t.nTw = (g.OW + sh.Wt - 1) / sh.Wt;
    t.rows = sh.rows;
    t.vec = sh.vec;
    t.a_bytes = (uint32_t)sh.rows * 128u;
    t.units = sh.mtiles * g.G * t.ntiles * c.split_k;
    t.fd_split = make_fastdiv((uint32_t)c.split_k);
    t.fd_gnt = make_fastdiv((uint32_t)(g.G * t.ntiles));
    t.fd_nTw = make_fastdiv((uint32_t)t.nTw);
    t.fd_nTh = make_fastdiv((uint32_t)t.nTh);
    t.fd_nTd = make_fastdiv((uint32_t)t.nTd);
    int err;
    switch (c.tile_n) {
      case 16: err = launch_tma_t<16>(g, c, t, tx, tm, s); break;
      case 32: err = launch_tma_t<32>(g, c, t, tx, tm, s); break;
      case 64: err = launch_tma_t<64>(g, c, t, tx, tm, s); break;
      case 128: err = launch_tma_t<128>(g, c, t, tx, tm, s); break;
      case 256: err = launch_tma_t<256>(g, c, t, tx, tm, s); break;
      default: return (int)cudaErrorInvalidValue;
    }
    if (err != 0 || c.split_k <= 1) return err;
    return launch_reduce(g, c, part, (const __half*)a.b, (const __half*)a.z, (__half*)a.y, s);
  }

  TcArgs ta;
  ta.x = (const uint16_t*)a.x;
  ta.b = (const __half*)a.b;
  ta.z = (const __half*)a.z;
  ta.y = (__half*)a.y;
  ta.part = part;
  ta.stages = c.stages;
  ta.chunks = (g.Kg + kBK - 1) / kBK;
  ta.chunks_per_split = (ta.chunks + c.split_k - 1) / c.split_k;
  ta.split = c.split_k;
  ta.ntiles = (g.Mg + c.tile_n - 1) / c.tile_n;
  ta.row_tiles = ((long long)g.N * g.P + kBM - 1) / kBM;
  ta.units = ta.row_tiles * g.G * ta.ntiles * c.split_k;
  ta.fd_split = make_fastdiv((uint32_t)c.split_k);
  ta.fd_gnt = make_fastdiv((uint32_t)(g.G * ta.ntiles));
  ta.fd_P = make_fastdiv((uint32_t)g.P);
  ta.fd_OW = make_fastdiv((uint32_t)g.OW);
  ta.fd_OH = make_fastdiv((uint32_t)g.OH);
  const int err = chan ? launch_bn<true>(g, c, ta, tm, s) : launch_bn<false>(g, c, ta, tm, s);
  if (err != 0 || c.split_k <= 1) return err;
  return launch_reduce(g, c, part, ta.b, ta.z, ta.y, s);
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
