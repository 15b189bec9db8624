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
// The weights are then read from a copy in that order, written into the workspace by the
// prologue launch, which also repacks X (channels innermost) for the A operand.
//
// Two persistent, warp-specialised kernels (one CTA per SM) share the MMA and epilogue
// design; they differ in how A reaches shared memory:
//   igemm_tma_kernel (C/group % 64 == 0): A is one 5-D TMA box of X repacked in 64-channel
//     blocks per chunk (TMA applies stride, dilation and zero padding); 10 warps: 8
//     epilogue, MMA, TMA producer.
//   igemm_tc_kernel (other C/group): A is gathered from a channels-last copy of X by two
//     sets of four gather warps that take alternate chunks (thread t of a set owns tile
//     row t, one output pixel, and issues one cp.async per valid 16/8/4-byte unit straight
//     into the 128-byte-swizzled K-major row); 26 warps: 16 epilogue, 8 gather, MMA, TMA
//     (weights).
// One lane of the MMA warp issues tcgen05.mma (M = 128, N = BN, K = 16) and tcgen05.commit
// into TMEM accumulators; the epilogue warps read them with tcgen05.ld (lane = pixel,
// column = channel), add B[m] and Z, apply the activation, round once to f16 and store
// NC(D)HW Y as 16-byte vectors through a per-warp staging tile. A ring of `stages`
// shared-memory chunks (A 16 KB + B BN*128 B each) with full/empty mbarriers connects the
// producers to the MMA; acc_full/acc_empty connect the MMA to the epilogue.
//
// Split-K (README variants implicit_im2col_tiled_reg_splitk: the reduction is
// partitioned when the unsplit grid is too small, raw partial sums are combined, and
// the bias and activation are applied once): a work unit is (tile, split); units of a
// split plan write raw f32 partials to the workspace and splitk_reduce_kernel adds the
// splits in a fixed order, then applies B, Z and the activation (deterministic).
//
// Every mbarrier wait is bounded in time (2 s); a wait that gives up sets a shared abort
// flag and the device error word, and the CTA stops issuing work, waits (with a limit of
// its own, ignoring the flag) for the MMAs and TMA loads it already issued, frees TMEM and
// exits.
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
constexpr int kWarps = 26;
constexpr int kThreads = kWarps * 32;
constexpr int kEpiWarp0 = 0;      // warps 0-15 (four per TMEM lane quarter)
constexpr int kEpiWarps = 16;
constexpr int kGatherWarp0 = 16;  // warps 16-23: two sets of four, one thread per tile row
constexpr int kGatherWarps = 8;
constexpr int kMmaWarp = 24;
constexpr int kTmaWarp = 25;
constexpr uint32_t kStagingBytes = 1024;  // per epilogue warp: [16 channels][32 pixels] f16
constexpr int kMaxStages = 8;
constexpr int kMaxTab = 1024;    // per-copy table entries of a GEMM row
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Shared-memory ring depth for a tile width: as many (A 16 KB + B) chunks as fit in
// 200 KB, at most kMaxStages, even (the two gather sets alternate chunks).
__host__ __device__ constexpr int stages_for(int bn) {
  const int st = (200 * 1024) / (kBM * kBK * 2 + bn * kBK * 2);
  const int capped = (st > kMaxStages ? kMaxStages : st) & ~1;
  return capped < 2 ? 2 : capped;
}
// Chunks whose copies a gather thread keeps in flight. Two gather sets take the chunks of
// even and odd sequence number; a set waiting for a free stage holds at most depth - 1
// chunks that are loaded but not yet handed to the MMA, all newer than 2 * depth chunks
// before the one it waits for. The stage it waits for was last used S chunks before: with
// S >= 2 * depth that chunk is older than every chunk either set still owes, so the wait
// never depends on an arrival a gather set still owes.
__host__ __device__ constexpr int gather_depth(int bn) { return stages_for(bn) / 2 < 4 ? stages_for(bn) / 2 : 4; }
constexpr unsigned kErrWaitTimeout = 1u;

struct TcArgs {
  const uint16_t* xc;   // X repacked channels-last: [G][N][pixel][cp]
  const __half* b;
  const __half* z;
  __half* y;
  float* part;          // split-K partials [split][N][M][P] (f32), or null
  int stages;
  int cp;               // channels per packed pixel: 2, 4 or C/group rounded up to 8
  int row_units;        // copies per GEMM row: KV (cp < 8, one tap each) or KV * cp / 8
  int upc;              // copies per 64-wide chunk: 8 (16 bytes), 16 (8 bytes), 32 (4 bytes)
  int chunks;           // ceil(KV * cp / 64)
  int chunks_per_split;
  int split;
  int ntiles;           // channel tiles per group
  long long row_tiles;  // ceil(N*P / 128)
  long long units;      // row_tiles * G * ntiles * split
  FastDiv fd_split, fd_gnt, fd_ntiles, fd_P, fd_OW, fd_OH;  // unit and pixel decoding
};

// TMEM accumulators of the gathered-A kernel: as many BN-column buffers as fit in the 512
// columns (at most 8), drained by `sets` groups of epilogue warps that take the tiles in
// turn, so that several tiles are in the epilogue at once.
template <int BN>
struct AccPlan {
  static constexpr uint32_t cols = BN < 32 ? 32 : BN;
  static constexpr int nacc = (512 / cols) > 8 ? 8 : (int)(512 / cols);
  static constexpr int sets = nacc >= 4 ? 4 : nacc;
  static constexpr uint32_t tmem_cols = (uint32_t)nacc * cols;  // a power of two
};
constexpr int kMaxAcc = 8;

struct SharedCtl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t acc_full[kMaxAcc];
  uint64_t acc_empty[kMaxAcc];
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

// Wait for operations this CTA has already issued (MMAs behind a commit, TMA loads behind an
// armed barrier). Issued operations always complete, so this wait ignores the abort flag and
// only stops at its own time limit (then it records the timeout and returns).
constexpr uint64_t kDrainLimitNs = 200000000ull;
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  if (ptx::mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (ptx::mbar_try_wait(bar, parity)) return;
    if ((i & 63u) == 0 && ptx::globaltimer_ns() - t0 > kDrainLimitNs) {
      atomicOr(&g_device_error, kErrWaitTimeout);
      return;
    }
  }
}

// A TMA producer that stops early (abort) waits for the loads it issued: chunks [0, armed)
// went to stage chunk % S with phase parity (chunk / S) & 1; a chunk whose phase already
// completed returns at once.
__device__ __forceinline__ void drain_armed(const uint64_t* full, uint32_t armed, int S) {
  const uint32_t s = (uint32_t)S;
  for (uint32_t j = armed > s ? armed - s : 0u; j < armed; ++j)
    drain_wait(ptx::smem_addr(&full[j % s]), (j / s) & 1u);
}

// Bit t set when tap t of an axis lands inside X: 0 <= i0 + t * d < n, for k <= 32 taps.
__device__ __forceinline__ uint32_t tap_mask(int i0, int d, int n, int k) {
  if (d == 1) {
    const int lo = i0 < 0 ? -i0 : 0;
    const int hi = min(k - 1, n - 1 - i0);
    if (hi < lo) return 0u;
    const uint32_t upto = hi >= 31 ? 0xffffffffu : (2u << hi) - 1u;
    return upto & ~((1u << lo) - 1u);
  }
  uint32_t m = 0;
  for (int t = 0; t < k; ++t) {
    const int v = i0 + t * d;
    if (v >= 0 && v < n) m |= 1u << t;
  }
  return m;
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
  t.grp = (int)fast_div(gct, a.fd_ntiles);
  t.ct = (int)gct - t.grp * a.ntiles;
  t.c_begin = t.sp * a.chunks_per_split;
  t.nk = min(a.chunks_per_split, a.chunks - t.c_begin);
  return t;
}

// ---------------------------------------------------------------- epilogue
// TMEM lane = output pixel, column = output channel. A warp owns one 32-lane quarter and
// every other 16-column group of the accumulator; per group it loads 16 f32 columns,
// adds B[m] and Z, applies the activation, rounds to f16 and stores NC(D)HW Y. In the
// vector path (P % 8 == 0) the 16 x 32 results go through the warp's staging tile
// [16 channels][32 pixels] so that Z and Y move as 16-byte vectors (8 pixels of one
// channel); otherwise each lane stores its own pixel's 16 channels.

// Where one tile's rows land in Y: this lane's pixel, and the 8-pixel group this lane
// moves in the vector path (lane l: pixels 8 (l % 4) .. 8 (l % 4) + 7 of its quarter).
struct EpiRows {
  bool row_ok;      // this lane's pixel exists
  long long obase;  // n * M * P + pixel index of this lane's pixel
  bool grp_ok;      // this lane's 8-pixel group exists
  long long gbase;  // n * M * P + first pixel of that group
};

// Z of channels mcb + lane / 4 and mcb + lane / 4 + 8 for this lane's pixel group.
__device__ __forceinline__ void load_z16(const __half* z, const EpiRows& er, int mcb, int m_end,
                                         long long P, int lane, uint4& z0, uint4& z1) {
  const int ch0 = lane >> 2, ch1 = ch0 + 8;
  const uint4 zero = make_uint4(0, 0, 0, 0);
  z0 = (er.grp_ok && mcb + ch0 < m_end) ? ptx::ldg_nc_v4(z + er.gbase + (long long)(mcb + ch0) * P)
                                        : zero;
  z1 = (er.grp_ok && mcb + ch1 < m_end) ? ptx::ldg_nc_v4(z + er.gbase + (long long)(mcb + ch1) * P)
                                        : zero;
}

// Activation of 16 pre-activation values and f16 rounding into this lane's column of the
// staging tile ys[16 channels][32 pixels] (plain shared-memory accesses, so the row
// offsets fold into the store instructions).
template <int ACT>
__device__ __forceinline__ void stage16(const float (&v)[16], __half* ys, int lane, float alpha,
                                        float beta) {
  float o[16];
#pragma unroll
  for (int jj = 0; jj < 16; ++jj) o[jj] = act_eval<ACT, true>(v[jj], alpha, beta);
#pragma unroll
  for (int jj = 0; jj < 16; jj += 2) {
    // one packed conversion for two channels, then the two 2-byte stores
    const __half2 h2 = __floats2half2_rn(o[jj], o[jj + 1]);
    ys[jj * 32 + lane] = __low2half(h2);
    ys[(jj + 1) * 32 + lane] = __high2half(h2);
  }
}

// ACT value of the split-K kernels' epilogue: raw f32 partial sums, nothing applied.
constexpr int kActPartial = -1;

// One tile's epilogue for this warp. acc = TMEM address of the warp's lane quarter in the
// tile's accumulator buffer; channels [m_first, m_first + BN) of the tile, of which those
// below m_end exist; the warp takes the 16-column groups c_first, c_first + c_step, ...;
// zn0/zn1 = Z of the warp's first group, already requested (vector path). With ACT == kActPartial, y is the f32 partial-sum array of this unit's split.
// Compute and staging are the same for both store paths, which differ only in how Z
// reaches the staging tile and how Y leaves it: the vector path moves 8-pixel groups as
// 16-byte vectors, the scalar path (P % 8 != 0) moves each lane's own pixel.
template <int BN, int ACT>
__device__ __forceinline__ void epilogue_tile(const ConvGeom& g, const __half* b, const __half* z,
                                              void* y, bool vec, const EpiRows& er, int m_first,
                                              int m_end, uint32_t acc, int c_first, int c_step,
                                              int lane, __half* ys, uint4 zn0, uint4 zn1) {
  const bool hz = z != nullptr, hb = b != nullptr;
  __half* zs = ys;  // Z passes through the same tile: each lane reads back only its own column
#pragma unroll 1
  for (int c0 = c_first; c0 < BN; c0 += c_step) {
    const int mcb = m_first + c0;
    if (mcb >= m_end) break;  // the same for the whole warp
    const int nvalid = min(16, m_end - mcb);
    if constexpr (ACT == kActPartial) {
      float v[16];
      __syncwarp();
      ptx::tmem_ld16(acc + (uint32_t)c0, v);
      if (er.row_ok) {
        float* pp = static_cast<float*>(y) + er.obase + (long long)mcb * g.P;
#pragma unroll
        for (int jj = 0; jj < 16; ++jj)
          if (jj < nvalid) pp[(long long)jj * g.P] = v[jj];
      }
      continue;
    } else {
      const uint4 zc0 = zn0, zc1 = zn1;
      if (vec && hz && c0 + c_step < BN) load_z16(z, er, mcb + c_step, m_end, g.P, lane, zn0, zn1);
      uint32_t bl = 0;  // bias of channel mcb + lane % 16, requested before the accumulator
      if (hb) bl = ptx::ld1_u16(b + mcb + (lane & 15), (lane & 15) < nvalid ? 1u : 0u);
      if (hz) {
        if (vec) {
          reinterpret_cast<uint4*>(zs)[(lane >> 2) * 4 + (lane & 3)] = zc0;
          reinterpret_cast<uint4*>(zs)[((lane >> 2) + 8) * 4 + (lane & 3)] = zc1;
        } else {
#pragma unroll
          for (int jj = 0; jj < 16; ++jj)
            zs[jj * 32 + lane] = __ushort_as_half((unsigned short)ptx::ld1_u16(
                z + er.obase + (long long)(mcb + jj) * g.P, (er.row_ok && jj < nvalid) ? 1u : 0u));
        }
      }
      float v[16];
      __syncwarp();
      ptx::tmem_ld16(acc + (uint32_t)c0, v);
      if (hb) {
#pragma unroll
        for (int jj = 0; jj < 16; ++jj)
          v[jj] += __half2float(__ushort_as_half((unsigned short)__shfl_sync(0xffffffffu, bl, jj)));
      }
      if (hz) {
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) v[jj] += __half2float(zs[jj * 32 + lane]);
      }
      stage16<ACT>(v, ys, lane, g.alpha, g.beta);
      __syncwarp();
      __half* yh = static_cast<__half*>(y);
      if (vec) {
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int ch = (lane >> 2) + 8 * t;
          if (er.grp_ok && ch < nvalid) {
            const uint4 yv = reinterpret_cast<const uint4*>(ys)[ch * 4 + (lane & 3)];
            ptx::st_global_v4(yh + er.gbase + (long long)(mcb + ch) * g.P, yv);
          }
        }
      } else if (er.row_ok) {
        for (int jj = 0; jj < nvalid; ++jj) yh[er.obase + (long long)(mcb + jj) * g.P] = ys[jj * 32 + lane];
      }
      __syncwarp();
    }
  }
}

// Epilogue warps of the gathered-A kernel: tile rows are 128 consecutive output pixels
// q = n * P + pixel.
template <int BN, int ACT>
__device__ __forceinline__ void gather_epilogue(const ConvGeom& g, const TcArgs& a, SharedCtl& ctl,
                                                uint32_t tmem, uint8_t* staging, int warp, int lane) {
  using AP = AccPlan<BN>;
  const int q4 = (warp - kEpiWarp0) & 3;  // TMEM lane quarter
  const int j = (warp - kEpiWarp0) >> 2;
  const int eset = j % AP::sets;          // takes tiles tcount = eset, eset + sets, ...
  constexpr int kWpq = 4 / AP::sets;      // warps of a set per lane quarter
  const int c_first = (j / AP::sets) * 16;  // 16-column groups c_first + 16 kWpq k
  const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
  // 16-byte Y/Z vectors need 8-pixel groups inside one image (P % 8 == 0)
  const bool vec = (g.P % 8) == 0;
  __half* ys = reinterpret_cast<__half*>(staging + (warp - kEpiWarp0) * kStagingBytes);
  const long long NP = (long long)g.N * g.P;
  const long long MP = (long long)g.M * g.P;
  volatile int* abort_flag = &ctl.abort_flag;
  uint32_t tcount = (uint32_t)eset;
  for (long long u = blockIdx.x + (long long)eset * gridDim.x; u < a.units;
       u += (long long)AP::sets * gridDim.x, tcount += AP::sets) {
    if (*abort_flag) break;
    const Unit un = decode_unit(u, a, g.G);
    const uint32_t b = tcount % (uint32_t)AP::nacc;
    EpiRows er;
    const long long q = un.rt * kBM + q4 * 32 + lane;
    er.row_ok = q < NP;
    er.obase = 0;
    if (er.row_ok) {
      const long long n = fast_div((uint32_t)q, a.fd_P);
      er.obase = n * MP + (q - n * g.P);
    }
    const long long gq = un.rt * kBM + q4 * 32 + (lane & 3) * 8;
    er.grp_ok = gq < NP;
    er.gbase = 0;
    if (er.grp_ok) {
      const long long gn = fast_div((uint32_t)gq, a.fd_P);
      er.gbase = gn * MP + (gq - gn * g.P);
    }
    const int m_first = un.grp * g.Mg + un.ct * BN, m_end = un.grp * g.Mg + g.Mg;
    void* out = a.y;
    if constexpr (ACT == kActPartial) out = a.part + (long long)un.sp * NP * g.M;
    uint4 zn0 = make_uint4(0, 0, 0, 0), zn1 = zn0;
    if (ACT != kActPartial && vec && a.z && m_first + c_first < m_end)
      load_z16(a.z, er, m_first + c_first, m_end, g.P, lane, zn0, zn1);
    if (!bounded_wait(ptx::smem_addr(&ctl.acc_full[b]), (tcount / AP::nacc) & 1, abort_flag)) break;
    ptx::tc_fence_after();
    epilogue_tile<BN, ACT>(g, a.b, a.z, out, vec, er, m_first, m_end, lane_base + b * AP::cols,
                           c_first, kWpq * 16, lane, ys, zn0, zn1);
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&ctl.acc_empty[b]));
  }
}

template <int BN, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
    igemm_tc_kernel(const ConvGeom g, const TcArgs a, const __grid_constant__ CUtensorMap tmap_w) {
  using AP = AccPlan<BN>;
  constexpr uint32_t kTmemCols = AP::tmem_cols;
  constexpr uint32_t kABytes = kBM * kBK * 2;   // 16 KB
  constexpr uint32_t kBBytes = BN * kBK * 2;
  constexpr uint32_t kStageBytes = kABytes + kBBytes;
  constexpr uint32_t kIdesc = ptx::idesc_f16_f32(kBM, BN);

  extern __shared__ uint8_t dsmem[];
  __shared__ SharedCtl ctl;
  // per copy unit p of a GEMM row (cp >= 8: tap p / (cp / 8), channels 8 (p % (cp / 8)) ..;
  // cp < 8: tap p, all cp channels): {offset from the row's first packed pixel in
  // elements, (ky * KW + kx) | kz << 8}; units past the end of K carry kz = 31, a bit that
  // no row's depth mask has
  __shared__ __align__(16) int2 tab[kMaxTab];

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t base = (ptx::smem_addr(dsmem) + 1023u) & ~1023u;
  const int S = a.stages;
  const long long NP = (long long)g.N * g.P;
  const int HW = g.IH * g.IW;

  const int cp8 = a.cp >= 8 ? a.cp / 8 : 1;
  for (int p = tid; p < a.chunks * a.upc && p < kMaxTab; p += kThreads) {
    if (p < a.row_units) {
      const int t = p / cp8, c8 = p - t * cp8;
      const int kx = t % g.KW, ky = (t / g.KW) % g.KH, kz = t / (g.KW * g.KH);
      tab[p] = make_int2((kz * g.dD * HW + ky * g.dH * g.IW + kx * g.dW) * a.cp + c8 * 8,
                         (ky * g.KW + kx) | (kz << 8));
    } else {
      tab[p] = make_int2(0, 31 << 8);
    }
  }
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(ptx::smem_addr(&ctl.full[s]), 4 + 1);  // 4 gather warps + TMA
      ptx::mbar_init(ptx::smem_addr(&ctl.empty[s]), 1);
    }
    for (int b = 0; b < AP::nacc; ++b) {
      ptx::mbar_init(ptx::smem_addr(&ctl.acc_full[b]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl.acc_empty[b]), kEpiWarps / AP::sets);
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
  // everything above touched no global memory; the prologue's outputs (and X, W, B, Z) are
  // read only after the previous kernel has completed
  ptx::pdl_wait();

  if (warp >= kGatherWarp0 && warp < kGatherWarp0 + kGatherWarps) {
    // ================================================================ A gather
    const uint32_t set = (uint32_t)(warp - kGatherWarp0) >> 2;  // takes chunks it % 2 == set
    const int r = ((warp - kGatherWarp0) & 3) * 32 + lane;       // tile row
    const uint32_t swz = (uint32_t)(r & 7);
    constexpr int kDepth = gather_depth(BN);
    // With a single chunk of K every stage always holds chunk 0, so the units past the end
    // of K are zero in every stage: they are written once here and skipped afterwards.
    const int pad_from = a.chunks == 1 ? a.row_units : INT_MAX;
    if (a.chunks == 1) {
      const int ub = a.upc == 8 ? 16 : a.upc == 16 ? 8 : 4;  // bytes per unit
      for (int st = (int)set; st < S; st += 2)
        for (int p = a.row_units; p < a.upc; ++p) {
          const uint32_t piece = (uint32_t)(p * ub) >> 4, off = (uint32_t)(p * ub) & 15u;
          const uint32_t dst = ((base + (uint32_t)st * kStageBytes + (uint32_t)r * 128u) | (swz << 4)) ^ (piece << 4);
          if (ub == 16) ptx::st_shared_v4(dst, 0u, 0u, 0u, 0u);
          else if (ub == 8) ptx::st_shared_v2(dst + off, 0u, 0u);
          else ptx::st_shared_u32(dst + off, 0u);
        }
    }
    uint32_t it = 0, last_it = 0;
    int pending = 0;  // own chunks whose copies are in flight, newest = last_it
    bool stop = false;
    for (long long u = blockIdx.x; u < a.units && !stop; u += gridDim.x) {
      if (*abort_flag) break;
      const Unit un = decode_unit(u, a, g.G);
      const int first = (int)((it & 1u) ^ set);  // this set's first chunk of the unit
      if (first >= un.nk) {
        it += (uint32_t)un.nk;
        continue;
      }
      // where this thread's row reads X: validity masks (bit kz of mz: depth tap kz lands
      // inside X; bit ky * KW + kx of mhw: the (ky, kx) tap does, KH * KW <= 64) and the
      // row's first packed pixel (possibly outside X: only valid taps are read)
      uint32_t mz = 0;
      uint64_t mhw = 0;
      const uint16_t* xg = a.xc;
      {
        const long long q = un.rt * kBM + r;
        if (q < NP) {
          uint32_t nn, o, t1, w1, h1;
          fast_divmod((uint32_t)q, a.fd_P, nn, o);
          fast_divmod(o, a.fd_OW, t1, w1);
          fast_divmod(t1, a.fd_OH, o, h1);
          const int iz0 = (int)o * g.sD - g.pD, iy0 = (int)h1 * g.sH - g.pH, ix0 = (int)w1 * g.sW - g.pW;
          mz = tap_mask(iz0, g.dD, g.ID, g.KD);
          const uint32_t mx = tap_mask(ix0, g.dW, g.IW, g.KW);
          const uint32_t my = tap_mask(iy0, g.dH, g.IH, g.KH);
          if (mx) {
            for (uint32_t m = my; m; m &= m - 1) mhw |= (uint64_t)mx << ((__ffs(m) - 1) * g.KW);
          }
          xg = a.xc + ((long long)(un.grp * g.N + (int)nn) * g.IS + ((iz0 * g.IH + iy0) * g.IW + ix0)) * a.cp;
        }
      }
      auto valid = [&](int bits) -> uint32_t {
        return (uint32_t)(mhw >> (bits & 0xff)) & (mz >> (bits >> 8)) & 1u;
      };
      for (int i = first; i < un.nk; i += 2) {
        const uint32_t itc = it + (uint32_t)i;
        const int s = (int)(itc % (uint32_t)S);
        if (itc >= (uint32_t)S &&
            !bounded_wait(ptx::smem_addr(&ctl.empty[s]), ((itc / S) - 1) & 1, abort_flag)) {
          stop = true;
          break;
        }
        // the chunk's units: one validity test and one asynchronous copy each, straight
        // into the 128-byte-swizzled row; invalid units (taps outside X, padding past K, rows
        // past N*P) are zeros written by plain shared stores
        const int4* tp = reinterpret_cast<const int4*>(&tab[(un.c_begin + i) * a.upc]);
        const uint32_t arow = (base + (uint32_t)s * kStageBytes + (uint32_t)r * 128u) | (swz << 4);
        if (a.upc == 8) {
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const int4 t2 = tp[h];
            const uint32_t d0 = arow ^ ((uint32_t)(2 * h) << 4), d1 = arow ^ ((uint32_t)(2 * h + 1) << 4);
            if (2 * h < pad_from) {
              if (valid(t2.y)) ptx::cp_async16(d0, xg + t2.x, 16u); else ptx::st_shared_v4(d0, 0u, 0u, 0u, 0u);
            }
            if (2 * h + 1 < pad_from) {
              if (valid(t2.w)) ptx::cp_async16(d1, xg + t2.z, 16u); else ptx::st_shared_v4(d1, 0u, 0u, 0u, 0u);
            }
          }
        } else if (a.upc == 16) {
          // two taps of 4 channels (8 bytes each) per 16-byte piece
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int4 t2 = tp[j];
            const uint32_t dst = arow ^ ((uint32_t)j << 4);
            if (2 * j < pad_from) {
              if (valid(t2.y)) ptx::cp_async8(dst, xg + t2.x, 8u); else ptx::st_shared_v2(dst, 0u, 0u);
            }
            if (2 * j + 1 < pad_from) {
              if (valid(t2.w)) ptx::cp_async8(dst + 8u, xg + t2.z, 8u); else ptx::st_shared_v2(dst + 8u, 0u, 0u);
            }
          }
        } else {
          // four taps of 2 channels (4 bytes each) per 16-byte piece
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint32_t dst = arow ^ ((uint32_t)j << 4);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int4 t2 = tp[2 * j + h];
              if (4 * j + 2 * h < pad_from) {
                if (valid(t2.y)) ptx::cp_async4(dst + 8u * h, xg + t2.x, 4u); else ptx::st_shared_u32(dst + 8u * h, 0u);
              }
              if (4 * j + 2 * h + 1 < pad_from) {
                if (valid(t2.w)) ptx::cp_async4(dst + 8u * h + 4u, xg + t2.z, 4u); else ptx::st_shared_u32(dst + 8u * h + 4u, 0u);
              }
            }
          }
        }
        ptx::cp_async_commit();
        last_it = itc;
        if (++pending == kDepth) {
          // this set's oldest chunk in flight (kDepth - 1 own chunks ago) has landed
          ptx::cp_async_wait<kDepth - 1>();
          ptx::fence_proxy_async_smem();
          __syncwarp();
          const uint32_t old = itc - 2u * (uint32_t)(kDepth - 1);
          if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&ctl.full[old % (uint32_t)S]));
          --pending;
        }
      }
      it += (uint32_t)un.nk;
    }
    // hand over the chunks still in flight (also after an abort: copies always complete)
    ptx::cp_async_wait<0>();
    ptx::fence_proxy_async_smem();
    __syncwarp();
    for (int k = pending - 1; k >= 0; --k) {
      const uint32_t old = last_it - 2u * (uint32_t)k;
      if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&ctl.full[old % (uint32_t)S]));
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
      if (*abort_flag) drain_armed(ctl.full, it, S);
    }
  } else if (warp == kMmaWarp) {
    // ================================================================ MMA issue
    if (lane == 0) {
      uint32_t it = 0, tcount = 0;
      for (long long u = blockIdx.x; u < a.units; u += gridDim.x, ++tcount) {
        if (*abort_flag) break;
        const Unit un = decode_unit(u, a, g.G);
        const uint32_t b = tcount % (uint32_t)AP::nacc;
        if (tcount >= (uint32_t)AP::nacc &&
            !bounded_wait(ptx::smem_addr(&ctl.acc_empty[b]), ((tcount / AP::nacc) - 1) & 1, abort_flag))
          break;
        ptx::tc_fence_after();
        const uint32_t dacc = tmem + b * AP::cols;
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
      drain_wait(ptx::smem_addr(&ctl.drain), 0);
    }
  } else {
    // ================================================================ epilogue (warps 0-15)
    // one loop per activation, chosen once: the group loop carries no dispatch
#define FCONV_EPI_LOOP(ACT) gather_epilogue<BN, ACT>(g, a, ctl, tmem, dsmem + (base - ptx::smem_addr(dsmem)) + (size_t)S * kStageBytes, warp, lane)
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
  if (warp == kMmaWarp) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}


// ============================================================================
// TMA-fed variant (C/group a multiple of 64). X is first repacked into blocks of 64
// channels, channels innermost: Xb[c/64][n][d][h][w][64] (prologue launch). A tile of
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
  FastDiv fd_split, fd_gnt, fd_ntiles, fd_nTw, fd_nTh, fd_nTd;
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
  t.grp = (int)fast_div(gct, a.fd_ntiles);
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

// Epilogue warps of the TMA-fed kernel: tile rows are the pixels of a box (Nb images x
// Dt x Ht x Wt), row r = ((nb * Dt + dt) * Ht + ht) * Wt + wt.
template <int BN, int ACT>
__device__ __forceinline__ void tma_epilogue(const ConvGeom& g, const TmaArgs& a, SharedCtl& ctl,
                                             uint32_t tmem, uint8_t* staging, int warp, int lane) {
  constexpr uint32_t kAccCols = BN < 32 ? 32 : BN;
  const int q = warp & 3;      // TMEM lane quarter
  const int half = warp >> 2;  // which alternate 16-column groups
  const int r = q * 32 + lane;
  const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
  __half* ys = reinterpret_cast<__half*>(staging + warp * kStagingBytes);
  // this row's place in the pixel box, and that of the 8-row group this lane moves
  const int wt = r % a.Wt, ht = (r / a.Wt) % a.Ht, dt = (r / (a.Wt * a.Ht)) % a.Dt;
  const int nb = r / (a.Wt * a.Ht * a.Dt);
  const int gr = q * 32 + (lane & 3) * 8;
  const int gwt = gr % a.Wt, ght = (gr / a.Wt) % a.Ht, gdt = (gr / (a.Wt * a.Ht)) % a.Dt;
  const int gnb = gr / (a.Wt * a.Ht * a.Dt);
  const long long NP = (long long)g.N * g.P;
  const long long MP = (long long)g.M * g.P;
  const bool vec = a.vec != 0;
  volatile int* abort_flag = &ctl.abort_flag;
  uint32_t tcount = 0;
  for (long long u = blockIdx.x; u < a.units; u += gridDim.x, ++tcount) {
    if (*abort_flag) break;
    const TmaUnit un = decode_tma_unit(u, a, g.G);
    const uint32_t b = tcount & 1u;
    EpiRows er;
    const int n = un.n0 + nb, od = un.od0 + dt, oh = un.oh0 + ht, ow = un.ow0 + wt;
    er.row_ok = r < a.rows && n < g.N && od < g.OD && oh < g.OH && ow < g.OW;
    er.obase = er.row_ok ? (long long)n * MP + ((long long)od * g.OH + oh) * g.OW + ow : 0;
    const int gn = un.n0 + gnb, god = un.od0 + gdt, goh = un.oh0 + ght, gow = un.ow0 + gwt;
    er.grp_ok = gr < a.rows && gn < g.N && god < g.OD && goh < g.OH && gow < g.OW;
    er.gbase = er.grp_ok ? (long long)gn * MP + ((long long)god * g.OH + goh) * g.OW + gow : 0;
    const int m_first = un.grp * g.Mg + un.ct * BN, m_end = un.grp * g.Mg + g.Mg;
    void* out = a.y;
    if constexpr (ACT == kActPartial) out = a.part + (long long)un.sp * NP * g.M;
    uint4 zn0 = make_uint4(0, 0, 0, 0), zn1 = zn0;
    if (ACT != kActPartial && vec && a.z && m_first + half * 16 < m_end)
      load_z16(a.z, er, m_first + half * 16, m_end, g.P, lane, zn0, zn1);
    if (!bounded_wait(ptx::smem_addr(&ctl.acc_full[b]), (tcount >> 1) & 1, abort_flag)) break;
    ptx::tc_fence_after();
    epilogue_tile<BN, ACT>(g, a.b, a.z, out, vec, er, m_first, m_end, lane_base + b * kAccCols,
                           half * 16, 32, lane, ys, zn0, zn1);
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&ctl.acc_empty[b]));
  }
}

template <int BN, bool SPLIT>
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
  ptx::pdl_wait();  // the repacked X and the weight copy come from the prologue launch

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
      if (*abort_flag) drain_armed(ctl.full, it, S);
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
      drain_wait(ptx::smem_addr(&ctl.drain), 0);
    }
  } else {
    // ================================================================ epilogue (warps 0-7)
#define FCONV_EPI_LOOP(ACT) tma_epilogue<BN, ACT>(g, a, ctl, tmem, dsmem + (base - ptx::smem_addr(dsmem)) + (size_t)S * kStageBytes, warp, lane)
    if constexpr (SPLIT) {
      FCONV_EPI_LOOP(kActPartial);
    } else {
      FCONV_ACT_SWITCH(g.act, FCONV_EPI_LOOP)
    }
#undef FCONV_EPI_LOOP
  }

  ptx::pdl_trigger();
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kTmaMmaWarp) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- prologue
// Everything the main kernel reads in a layout of its own is written by ONE launch,
// prologue_kernel: its first `wblocks` blocks write the weight copy (one output channel
// each), the others repack X. Both parts only move data.

// X (N, C, spatial S) -> Xb[c/64][n][s][64]. Block (x, cb) moves 64 channels of the
// flattened positions q = n*S + s in [128x, 128x + 128), across image boundaries when S is
// small: four 16-byte loads per thread (8 positions of one channel), all in flight, into a
// shared tile, then four 16-byte stores per thread (8 channels of one position). Needs
// S % 8 == 0 (a load never straddles two images) and N*S < 2^31 (32-bit position
// decoding); otherwise pack_x_scalar is used.
constexpr int kPackPitch = 138;  // halves per channel row: 16-byte rows, few bank conflicts
constexpr size_t kPackSmem = 64 * kPackPitch * 2;

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
    uint32_t* d = reinterpret_cast<uint32_t*>(t + c * kPackPitch + pv * 8);  // 4-byte aligned
    d[0] = buf[i].x; d[1] = buf[i].y; d[2] = buf[i].z; d[3] = buf[i].w;
  }
  __syncthreads();
  uint16_t* dst = xb + ((long long)cb * NS + q0) * 64;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int o = threadIdx.x + 256 * i;
    const int p = o >> 3, part = o & 7;
    if (p >= rows) continue;
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      w[e] = (uint32_t)t[(8 * part + 2 * e) * kPackPitch + p] |
             ((uint32_t)t[(8 * part + 2 * e + 1) * kPackPitch + p] << 16);
    *reinterpret_cast<uint4*>(dst + (long long)p * 64 + 8 * part) = make_uint4(w[0], w[1], w[2], w[3]);
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

// X for the gather: Xc[g][n][pixel][cp], channels innermost, zero past C/group, so that
// each 16-byte piece of a GEMM row is one aligned load. One thread per packed pixel
// (plane gn = g * N + n from `by` in steps of `ny`): the reads of each channel plane are
// coalesced across the warp, and the warp's 16-byte writes cover one run of Xc.
__device__ __forceinline__ void pack_cl(const uint16_t* __restrict__ x, uint16_t* __restrict__ xc,
                                        int N, int G, int Cg, int cp, int S, int bx, int nx,
                                        int by, int ny) {
  for (int gn = by; gn < G * N; gn += ny) {
    const int gi = gn / N, n = gn - gi * N;
    const uint16_t* src = x + ((long long)n * G + gi) * Cg * (long long)S;
    uint16_t* dst = xc + (long long)gn * S * cp;
    for (int sp = bx * 256 + threadIdx.x; sp < S; sp += nx * 256) {
      if (cp < 8) {  // 2 or 4 channels per pixel
        for (int c = 0; c < cp; ++c) dst[(long long)sp * cp + c] = c < Cg ? src[(long long)c * S + sp] : (uint16_t)0;
        continue;
      }
      for (int c8 = 0; c8 < cp; c8 += 8) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int c = c8 + 2 * e;
          const uint32_t lo = c < Cg ? (uint32_t)src[(long long)c * S + sp] : 0u;
          const uint32_t hi = c + 1 < Cg ? (uint32_t)src[(long long)(c + 1) * S + sp] : 0u;
          w[e] = lo | (hi << 16);
        }
        *reinterpret_cast<uint4*>(dst + (long long)sp * cp + c8) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }
}

// As pack_cl for S % 8 == 0: one work item per (plane gn, 8-channel group, 8 consecutive
// pixels j), items spread over the whole grid (item i of `items`, grid-stride from bi in
// steps of nb). Eight 16-byte loads (8 pixels of one channel plane each, coalesced across
// the warp), an 8 x 8 transpose of 16-bit values in registers (byte permutes: pixel 2k
// takes the low halves of word k of each channel pair, pixel 2k + 1 the high halves), eight
// 16-byte stores (8 channels of one pixel each).
__device__ __forceinline__ void pack_cl8(const uint16_t* __restrict__ x, uint16_t* __restrict__ xc,
                                         int N, int G, int Cg, int cp, int S, long long bi,
                                         long long nb) {
  const int S8 = S / 8;
  const int groups = cp >= 8 ? cp / 8 : 1;
  const long long items = (long long)G * N * groups * S8;
  for (long long it = bi * 256 + threadIdx.x; it < items; it += nb * 256) {
    // 32-bit decoding (the host keeps items below 2^31 on this path)
    const uint32_t rest = (uint32_t)it / (uint32_t)S8;
    const int j = (int)((uint32_t)it - rest * (uint32_t)S8);
    const int c8 = (int)(rest % (uint32_t)groups) * 8;
    const int gn = (int)(rest / (uint32_t)groups);
    const int gi = gn / N, n = gn - gi * N;
    const uint16_t* src = x + ((long long)n * G + gi) * Cg * (long long)S;
    uint16_t* dst = xc + (long long)gn * S * cp;
    if (cp < 8) {
      // 2 or 4 channels per pixel: the same transpose, keeping the first cp channels
      uint32_t w[4][4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint4 r = make_uint4(0, 0, 0, 0);
        if (c < Cg && c < cp) r = ptx::ldg_nc_v4(src + (long long)c * S + 8LL * j);
        w[c][0] = r.x; w[c][1] = r.y; w[c][2] = r.z; w[c][3] = r.w;
      }
      // the item's 8 pixels are 8 * cp contiguous elements: 16-byte stores
      uint32_t a0[4], a1[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        a0[k] = __byte_perm(w[0][k], w[1][k], 0x5410);  // pixel 2k, channels 0-1
        a1[k] = __byte_perm(w[0][k], w[1][k], 0x7632);  // pixel 2k + 1
      }
      if (cp == 2) {
#pragma unroll
        for (int h = 0; h < 2; ++h)
          ptx::st_global_v4(dst + (8LL * j + 4 * h) * 2,
                            make_uint4(a0[2 * h], a1[2 * h], a0[2 * h + 1], a1[2 * h + 1]));
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t b0 = __byte_perm(w[2][k], w[3][k], 0x5410), b1 = __byte_perm(w[2][k], w[3][k], 0x7632);
          ptx::st_global_v4(dst + (8LL * j + 2 * k) * 4, make_uint4(a0[k], b0, a1[k], b1));
        }
      }
      continue;
    }
    uint32_t w[8][4];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      uint4 r = make_uint4(0, 0, 0, 0);
      if (c8 + c < Cg) r = ptx::ldg_nc_v4(src + (long long)(c8 + c) * S + 8LL * j);
      w[c][0] = r.x; w[c][1] = r.y; w[c][2] = r.z; w[c][3] = r.w;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 lo = make_uint4(__byte_perm(w[0][k], w[1][k], 0x5410), __byte_perm(w[2][k], w[3][k], 0x5410),
                                  __byte_perm(w[4][k], w[5][k], 0x5410), __byte_perm(w[6][k], w[7][k], 0x5410));
      const uint4 hi = make_uint4(__byte_perm(w[0][k], w[1][k], 0x7632), __byte_perm(w[2][k], w[3][k], 0x7632),
                                  __byte_perm(w[4][k], w[5][k], 0x7632), __byte_perm(w[6][k], w[7][k], 0x7632));
      ptx::st_global_v4(dst + (8LL * j + 2 * k) * cp + c8, lo);
      ptx::st_global_v4(dst + (8LL * j + 2 * k + 1) * cp + c8, hi);
    }
  }
}

// Weights in the GEMM's K order, zero padded to kpad columns: wp[m][k'] for k' < kpad.
// One block per output channel: the row is staged in shared memory (16-byte loads when
// rows are 16-byte aligned), then each thread writes 8 consecutive k' as one 16-byte
// store, reading the permuted sources from shared memory.
//   block64 (TMA-fed A, C/group a multiple of 64): k' = (64-channel block, tap, channel)
//   otherwise (gathered A): k' = tap * cp + channel, zero for channels >= C/group
__device__ __forceinline__ int prep_src(int k, int Cg, int KV, int cp, int block64) {
  if (block64) {
    if (k >= Cg * KV) return -1;
    const int cb = k / (64 * KV), rem = k - cb * 64 * KV;
    const int tap = rem >> 6;
    return (cb * 64 + (rem & 63)) * KV + tap;
  }
  const int tap = k / cp, c = k - tap * cp;
  return (c < Cg && tap < KV) ? c * KV + tap : -1;
}

__device__ __forceinline__ void prep_weights_row(const uint16_t* __restrict__ w, uint16_t* __restrict__ wp,
                                                 int m, int Cg, int KV, int kpad, int cp, int block64,
                                                 uint16_t* row) {
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
      const int src_k = prep_src(v * 8 + j, Cg, KV, cp, block64);
      e[j] = src_k >= 0 ? (uint32_t)row[src_k] : 0u;
    }
    reinterpret_cast<uint4*>(dst)[v] =
        make_uint4(e[0] | (e[1] << 16), e[2] | (e[3] << 16), e[4] | (e[5] << 16), e[6] | (e[7] << 16));
  }
}

enum PackKind { kPackBlock64 = 0, kPackBlock64Scalar = 1, kPackCl8 = 2, kPackCl = 3 };

struct PrologueArgs {
  const uint16_t* w;
  uint16_t* wp;         // weight copy, or null (no weight blocks)
  int wblocks;          // = M when wp, else 0
  int Cg, KV, kpad, cp, block64;
  const uint16_t* x;
  uint16_t* xp;
  int kind;             // PackKind
  int N, C, G;
  long long S;
  long long nx;         // pack blocks along the position axis
  int ny;               // pack blocks along the channel-block / plane axis
};

__global__ void __launch_bounds__(256) prologue_kernel(const PrologueArgs p) {
  extern __shared__ __align__(16) uint16_t psm[];
  ptx::pdl_trigger();  // the main kernel may set itself up meanwhile
  ptx::pdl_wait();     // X and W may be the previous kernel's outputs
  long long b = blockIdx.x;
  if (b < p.wblocks) {
    prep_weights_row(p.w, p.wp, (int)b, p.Cg, p.KV, p.kpad, p.cp, p.block64, psm);
    return;
  }
  b -= p.wblocks;
  const long long bx = b % p.nx;
  const int by = (int)(b / p.nx);
  switch (p.kind) {
    case kPackBlock64: pack_x_block(p.x, p.xp, p.N, p.C, p.S, bx, by, psm); break;
    case kPackBlock64Scalar: pack_x_scalar(p.x, p.xp, p.N, p.C, p.S, bx, p.nx); break;
    case kPackCl8: pack_cl8(p.x, p.xp, p.N, p.G, p.Cg, p.cp, (int)p.S, bx, p.nx); break;
    default: pack_cl(p.x, p.xp, p.N, p.G, p.Cg, p.cp, (int)p.S, (int)bx, (int)p.nx, by, p.ny); break;
  }
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

// Channels per packed pixel of the gathered A operand.
// (2 and 4 keep the zero padding of 1-4 channel inputs small: their copies are 4 or 8 bytes)
int cp_of(const ConvGeom& g) { return g.Cg <= 2 ? 2 : g.Cg <= 4 ? 4 : (g.Cg + 7) / 8 * 8; }
// Copy units of a GEMM row and per 64-wide chunk.
int units_of(const ConvGeom& g) { return cp_of(g) >= 8 ? g.KV * (cp_of(g) / 8) : g.KV; }
int upc_of(const ConvGeom& g) { return cp_of(g) >= 8 ? 8 : 64 / cp_of(g); }

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

template <int BN, bool SPLIT>
int launch_t(const ConvGeom& g, const IgemmConfig& c, const TcArgs& ta, const CUtensorMap& tm,
             cudaStream_t s) {
  // the gather's in-flight depth is sized for this ring (no wait on a chunk it still owes)
  if (c.stages < 2 * gather_depth(BN)) return (int)cudaErrorInvalidValue;
  const size_t smem = igemm_tc_smem_bytes(BN, c.stages);
  cudaError_t e = cudaFuncSetAttribute(igemm_tc_kernel<BN, SPLIT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int)e;
  return launch_pdl(igemm_tc_kernel<BN, SPLIT>, dim3((unsigned)c.grid), dim3(kThreads), smem, s, g,
                    ta, tm);
}

template <bool SPLIT>
int launch_bn(const ConvGeom& g, const IgemmConfig& c, const TcArgs& ta, const CUtensorMap& tm,
              cudaStream_t s) {
  switch (c.tile_n) {
    case 16: return launch_t<16, SPLIT>(g, c, ta, tm, s);
    case 32: return launch_t<32, SPLIT>(g, c, ta, tm, s);
    case 64: return launch_t<64, SPLIT>(g, c, ta, tm, s);
    case 128: return launch_t<128, SPLIT>(g, c, ta, tm, s);
    case 256: return launch_t<256, SPLIT>(g, c, ta, tm, s);
    default: return (int)cudaErrorInvalidValue;
  }
}

template <int BN, bool SPLIT>
int launch_tma_t(const ConvGeom& g, const IgemmConfig& c, const TmaArgs& t, const CUtensorMap& tx,
                 const CUtensorMap& tw, cudaStream_t s) {
  const size_t smem = (size_t)c.stages * (size_t)(kBM * kBK * 2 + BN * kBK * 2) + 1024 +
                      (size_t)kTmaEpiWarps * kStagingBytes;
  cudaError_t e = cudaFuncSetAttribute(igemm_tma_kernel<BN, SPLIT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int)e;
  return launch_pdl(igemm_tma_kernel<BN, SPLIT>, dim3((unsigned)c.grid), dim3(kTmaThreads), smem,
                    s, g, t, tx, tw);
}

int launch_reduce(const ConvGeom& g, const IgemmConfig& c, const float* part, const __half* b,
                  const __half* z, __half* y, cudaStream_t s) {
  const long long total = (long long)g.N * g.M * g.P;
  long long blocks = (total + 255) / 256;
  if (blocks > 152LL * 32) blocks = 152LL * 32;
  int err = 0;
#define FCONV_REDUCE(ACT)                                                                  \
  err = launch_pdl(splitk_reduce_kernel<ACT>, dim3((unsigned)blocks), dim3(256), 0, s, g, part, \
                   c.split_k, b, z, y, total)
  FCONV_ACT_SWITCH(g.act, FCONV_REDUCE)
#undef FCONV_REDUCE
  return err;
}

}  // namespace

int igemm_tc_stages(int tile_n) { return stages_for(tile_n); }

size_t igemm_tc_smem_bytes(int tile_n, int stages) {
  // operand ring + 1 KB alignment slack + the epilogue warps' Y/Z staging tiles
  return (size_t)stages * (size_t)(kBM * kBK * 2 + tile_n * kBK * 2) + 1024 + kEpiWarps * kStagingBytes;
}

// Weight copy in GEMM order (when W itself cannot be read by TMA in that order): the
// TMA-fed path needs it unless the kernel is 1x1 (then W's order is the block order);
// the gather path unless also C/group is a multiple of 8 (no channel padding, rows of
// whole 16-byte units).
static bool needs_prep(const ConvGeom& g, bool tma) {
  if (tma) return g.KV != 1;
  return !(g.KV == 1 && cp_of(g) == g.Cg && g.Cg % 8 == 0);  // TMA rows: 16-byte multiples
}

// Columns of the GEMM's K (the weight copy's row length when there is one).
static size_t kpad_of(const ConvGeom& g, bool tma) {
  return tma ? (size_t)g.Kg : round_up((size_t)g.KV * (size_t)cp_of(g), 8);
}

static size_t prep_bytes(const ConvGeom& g, bool tma) {
  return needs_prep(g, tma) ? round_up((size_t)g.M * kpad_of(g, tma) * 2, 1024) : 0;
}

// Repacked X: 64-channel blocks for the TMA-fed path, channels-last for the gather.
static size_t pack_bytes(const ConvGeom& g, bool tma) {
  const size_t pix = (size_t)g.N * (size_t)g.IS;
  return round_up(tma ? pix * (size_t)g.C * 2 : pix * (size_t)g.G * (size_t)cp_of(g) * 2, 1024);
}

size_t igemm_tc_workspace_bytes(const ConvGeom& g, const IgemmConfig& c) {
  const bool tma = use_tma(g, c.a_path);
  size_t b = prep_bytes(g, tma) + pack_bytes(g, tma);
  if (c.split_k > 1) b += (size_t)c.split_k * (size_t)g.N * (size_t)g.M * (size_t)g.P * 4;
  return b;
}

bool igemm_tc_tma_capable(const ConvGeom& g) { return tma_shape(g).ok; }

int igemm_tc_launches(const ConvGeom& g, const IgemmConfig& c) {
  (void)g;
  return 2 + (c.split_k > 1 ? 1 : 0);  // prologue, main kernel, split-K reduce
}

long long igemm_tc_mtiles(const ConvGeom& g, int a_path) {
  if (use_tma(g, a_path)) return tma_shape(g).mtiles;
  return ((long long)g.N * g.P + kBM - 1) / kBM;
}

int igemm_tc_chunks(const ConvGeom& g, int a_path) {
  return (int)((kpad_of(g, use_tma(g, a_path)) + kBK - 1) / kBK);
}

bool igemm_tc_gather_capable(const ConvGeom& g) {
  // validity masks: depth taps in 32 bits with bit 31 free, (ky, kx) taps in 64 bits
  if (g.KD > 31 || g.KH > 32 || g.KW > 32 || (long long)g.KH * g.KW > 64) return false;
  if (round_up((size_t)units_of(g), (size_t)upc_of(g)) > (size_t)kMaxTab) return false;
  // tap and row offsets (in packed elements, padded taps included) stay in 32-bit ints
  const long long span = (long long)(g.ID + g.pD + 1) * (g.IH + g.pH + 1) * (g.IW + g.pW + 1);
  if (span * cp_of(g) > INT_MAX / 2) return false;
  if ((long long)g.M * (long long)kpad_of(g, false) > INT_MAX) return false;
  return true;
}

bool igemm_tc_supported(const ConvGeom& g) {
  if (g.dtype != FCONV_F16) return false;
  if ((size_t)g.Kg * 2 > 200 * 1024) return false;  // weight row staged in shared memory
  // unit and pixel indices are decoded in 32 bits (every unit count is at most N*P*M)
  if ((long long)g.N * g.P * g.M >= 0x7fffffffLL) return false;
  return igemm_tc_gather_capable(g) || tma_shape(g).ok;
}

int launch_igemm_tc(const ConvGeom& g, const IgemmConfig& c, const ConvArgs& a, void* stream) {
  cudaStream_t s = (cudaStream_t)stream;
  if (c.stages < 2 || c.stages > kMaxStages || (c.stages & 1)) return (int)cudaErrorInvalidValue;
  EncodeTiledFn enc = encode_fn();
  if (!enc) return (int)cudaErrorNotSupported;
  const bool tma = use_tma(g, c.a_path);
  uint8_t* ws = (uint8_t*)a.ws;
  const size_t pb = prep_bytes(g, tma);
  const int kpad = (int)kpad_of(g, tma);
  const int cp = cp_of(g);
  // one prologue launch: the weight copy (when the GEMM's K order is not W's) and X
  // repacked for the A operand
  const size_t xb_bytes = pack_bytes(g, tma);
  uint16_t* xpack = (uint16_t*)(ws + pb);
  {
    PrologueArgs pa;
    pa.w = (const uint16_t*)a.w;
    pa.wp = pb ? (uint16_t*)ws : nullptr;
    pa.wblocks = pb ? g.M : 0;
    pa.Cg = g.Cg;
    pa.KV = g.KV;
    pa.kpad = kpad;
    pa.cp = cp;
    pa.block64 = tma ? 1 : 0;
    pa.x = (const uint16_t*)a.x;
    pa.xp = xpack;
    pa.N = g.N;
    pa.C = g.C;
    pa.G = g.G;
    pa.S = g.IS;
    size_t smem = pb ? (size_t)g.Kg * 2 : 0;
    long long pack_blocks;
    if (tma) {
      const long long NS = (long long)g.N * g.IS;
      if (g.IS % 8 == 0 && NS < 0x7fffff00LL) {
        pa.kind = kPackBlock64;
        pa.nx = (NS + 127) / 128;
        pa.ny = g.C / 64;
        pack_blocks = pa.nx * pa.ny;
        if (smem < kPackSmem) smem = kPackSmem;
      } else {
        pa.kind = kPackBlock64Scalar;
        long long blocks = (NS * (g.C / 8) + 255) / 256;
        if (blocks > 152LL * 32) blocks = 152LL * 32;
        pa.nx = blocks;
        pa.ny = 1;
        pack_blocks = blocks;
      }
    } else {
      const long long planes = (long long)g.G * g.N;
      pa.ny = (int)(planes < 65535 ? planes : 65535);
      const long long items = planes * (cp >= 8 ? cp / 8 : 1) * (g.IS / 8);
      if (g.IS % 8 == 0 && items + 152LL * 16 * 256 < 0x7fffffffLL) {
        // one item per (plane, 8-channel group, 8 pixels); enough blocks to fill the GPU
        pa.kind = kPackCl8;
        long long nb = (items + 255) / 256;
        if (nb > 152LL * 16) nb = 152LL * 16;
        pa.nx = nb;
        pa.ny = 1;
      } else {
        pa.kind = kPackCl;
        pa.nx = (g.IS + 255) / 256;
      }
      pack_blocks = pa.nx * pa.ny;
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
    t.fd_ntiles = make_fastdiv((uint32_t)t.ntiles);
    t.fd_nTw = make_fastdiv((uint32_t)t.nTw);
    t.fd_nTh = make_fastdiv((uint32_t)t.nTh);
    t.fd_nTd = make_fastdiv((uint32_t)t.nTd);
    int err;
    const bool sp = c.split_k > 1;
    switch (c.tile_n) {
      case 16: err = sp ? launch_tma_t<16, true>(g, c, t, tx, tm, s) : launch_tma_t<16, false>(g, c, t, tx, tm, s); break;
      case 32: err = sp ? launch_tma_t<32, true>(g, c, t, tx, tm, s) : launch_tma_t<32, false>(g, c, t, tx, tm, s); break;
      case 64: err = sp ? launch_tma_t<64, true>(g, c, t, tx, tm, s) : launch_tma_t<64, false>(g, c, t, tx, tm, s); break;
      case 128: err = sp ? launch_tma_t<128, true>(g, c, t, tx, tm, s) : launch_tma_t<128, false>(g, c, t, tx, tm, s); break;
      case 256: err = sp ? launch_tma_t<256, true>(g, c, t, tx, tm, s) : launch_tma_t<256, false>(g, c, t, tx, tm, s); break;
      default: return (int)cudaErrorInvalidValue;
    }
    if (err != 0 || c.split_k <= 1) return err;
    return launch_reduce(g, c, part, (const __half*)a.b, (const __half*)a.z, (__half*)a.y, s);
  }

  TcArgs ta;
  ta.xc = xpack;
  ta.b = (const __half*)a.b;
  ta.z = (const __half*)a.z;
  ta.y = (__half*)a.y;
  ta.part = part;
  ta.stages = c.stages;
  ta.cp = cp;
  ta.row_units = units_of(g);
  ta.upc = upc_of(g);
  ta.chunks = (kpad + kBK - 1) / kBK;
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
  ta.fd_ntiles = make_fastdiv((uint32_t)ta.ntiles);
  const int err = c.split_k > 1 ? launch_bn<true>(g, c, ta, tm, s) : launch_bn<false>(g, c, ta, tm, s);
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
