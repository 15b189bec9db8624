// Pieces shared by the tcgen05 implicit-GEMM kernels (k_igemm_tc.cu, k_igemm_patch.cu):
// tile constants, time-bounded mbarrier waits, the TMEM accumulator plan, the box tiling
// of output pixels and the fused epilogue of one tile.
//
// GEMM view per group g (the package's implicit im2col routes, README variants
// implicit_im2col_tiled_reg / implicit_im2col_subgroup_matrix), computed transposed so that
// the accumulator is channel-major:
//   D[m, p] = sum_k W[m, k] * A[p, k]
//   m = output channel of the group, 128 per tile (MMA M; TMEM lane = channel)
//   p = output pixel of a box of Nb images x Dt x Ht x Wt, at most 256 (MMA N; TMEM column)
//   k over (ci, tap), Kg = C/group * prod(kernel), consumed 64 per chunk
// The weights are the MMA's A operand and the im2col rows of the pixels its B operand, both
// K-major in 128-byte-swizzled shared memory. The epilogue reads 16 consecutive pixels of one
// channel per thread with tcgen05.ld, adds B[m] and Z, applies the activation in f32, rounds
// once to f16 and stores NC(D)HW Y as 16-byte vectors (8 pixels of one channel) straight from
// registers.
//
// Everything here has internal linkage: each translation unit that includes it gets its own
// copy, including its own device error word (read by fconv_check_device).
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "epilogue.cuh"
#include "fastdiv.cuh"
#include "fconv_internal.h"
#include "ptx.cuh"

namespace fconv {
namespace {

constexpr int kMT = 128;                  // MMA M: output channels per tile
constexpr int kMaxPx = 256;               // MMA N at most: output pixels per tile
constexpr int kBK = 64;                   // K per chunk: one 128-byte swizzled operand row
constexpr uint32_t kWBytes = kMT * kBK * 2;  // one chunk of the weights tile
constexpr int kMaxStages = 8;
constexpr int kMaxAcc = 8;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint64_t kDrainLimitNs = 200000000ull;
constexpr unsigned kErrWaitTimeout = 1u;
constexpr int kActPartial = -1;           // epilogue ACT of split-K units: raw f32 partials

// Set when a bounded wait of a kernel in this translation unit gives up.
__device__ unsigned g_tc_error = 0;

// Wait for phase `parity` of an mbarrier, for at most kWaitLimitNs. Gives up early when
// another warp of the CTA already gave up (abort_flag); a wait that runs out sets the flag
// and the device error word.
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
        atomicOr(&g_tc_error, kErrWaitTimeout);
        return false;
      }
    }
  }
}

// Wait for operations this CTA has already issued (MMAs behind a commit, TMA loads behind an
// armed barrier). Issued operations always complete, so this wait ignores the abort flag and
// only stops at its own time limit (then it records the timeout and returns).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  if (ptx::mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (ptx::mbar_try_wait(bar, parity)) return;
    if ((i & 63u) == 0 && ptx::globaltimer_ns() - t0 > kDrainLimitNs) {
      atomicOr(&g_tc_error, kErrWaitTimeout);
      return;
    }
  }
}

// A TMA producer that stops early (abort) waits for the loads it issued: loads [0, armed)
// went to slot j % S of `full` with phase parity (j / S) & 1; a load whose phase already
// completed returns at once.
__device__ __forceinline__ void drain_armed(const uint64_t* full, uint32_t armed, int S) {
  const uint32_t s = (uint32_t)S;
  for (uint32_t j = armed > s ? armed - s : 0u; j < armed; ++j)
    drain_wait(ptx::smem_addr(&full[j % s]), (j / s) & 1u);
}

// TMEM accumulators: as many NPX-column buffers as fit in the 512 columns (at most 8),
// drained by `sets` groups of epilogue warps (each group covering the four TMEM lane
// quarters) that take the tiles in turn, so that several tiles are in the epilogue at once.
// EPI = epilogue warps; each set has EPI / sets warps, EPI / (4 sets) per lane quarter.
template <int NPX, int EPI>
struct AccPlan {
  static constexpr uint32_t cols = NPX;
  static constexpr int nacc = (512 / NPX) > 8 ? 8 : 512 / NPX;
  static constexpr int sets = nacc < EPI / 4 ? nacc : EPI / 4;
  static constexpr int wpq = EPI / 4 / sets;
  static constexpr uint32_t tmem_cols = (uint32_t)nacc * cols;  // a power of two
  static_assert(sets * wpq * 4 == EPI, "epilogue warps cover the sets and quarters");
};

// ------------------------------------------------------------------ box tiling of pixels

// A tile's pixels are the output pixels of a box: Nb images x Dt x Ht x Wt (at most 256, or
// R sub-boxes of npx pixels each when the accumulator stacks R bands of channels);
// pixel i = ((nb * Dt + dt) * Ht + ht) * Wt + wt. A work unit is (box, group, channel tile,
// K split); unit u decodes as u = ((box * G + grp) * ntiles + ct) * split + sp.
struct BoxTiling {
  int G;                    // groups
  int Nb, Dt, Ht, Wt;
  int rows;                 // pixels of a box, Nb * Dt * Ht * Wt <= R * npx
  int nTd, nTh, nTw;        // boxes along depth, height, width
  int vec;                  // 8-pixel groups are 16-byte aligned runs of Y (P % 8 == 0)
  int ntiles;               // channel tiles of 128 per group
  int R, Mp, npx;           // accumulator bands: R sub-boxes of npx pixels, each with Mp
                            // lanes of channels (R = 128 / Mp; R = 1 unless Mg <= 64)
  int split, chunks, chunks_per_split;
  long long units;
  FastDiv fd_split, fd_gnt, fd_ntiles, fd_nTw, fd_nTh, fd_nTd;
};

struct BoxUnit {
  int n0, od0, oh0, ow0;
  int grp, ct, sp, c_begin, nk;
};

__device__ __forceinline__ BoxUnit decode_box_unit(long long u, const BoxTiling& t) {
  BoxUnit b;
  uint32_t r, sp, gct, rt, tw, th, td;
  fast_divmod((uint32_t)u, t.fd_split, r, sp);
  fast_divmod(r, t.fd_gnt, rt, gct);
  b.sp = (int)sp;
  b.grp = (int)fast_div(gct, t.fd_ntiles);
  b.ct = (int)gct - b.grp * t.ntiles;
  fast_divmod(rt, t.fd_nTw, rt, tw);
  fast_divmod(rt, t.fd_nTh, rt, th);
  fast_divmod(rt, t.fd_nTd, rt, td);
  b.n0 = (int)rt * t.Nb;
  b.od0 = (int)td * t.Dt;
  b.oh0 = (int)th * t.Ht;
  b.ow0 = (int)tw * t.Wt;
  b.c_begin = b.sp * t.chunks_per_split;
  b.nk = min(t.chunks_per_split, t.chunks - b.c_begin);
  return b;
}

// Position in a ring of n slots: the slot and the phase parity of its current use, advanced
// without division. A consumer waits for phase `phase` of a slot's full barrier; a producer
// waits for phase `phase ^ 1` of its empty barrier, which a fresh barrier reports complete.
struct Ring {
  uint32_t idx, phase;
  __device__ __forceinline__ void next(uint32_t n) {
    if (++idx == n) {
      idx = 0;
      phase ^= 1u;
    }
  }
};

// Walks the work units u = first, first + stride, ... of a CTA, keeping the unit's digits
// (least significant first: split, channel tile, group, box column, box row, box slice, image
// block) current with additions and carries instead of divisions.
struct UnitIter {
  long long u, stride;
  int sp, ct, grp, tw, th, td, nb;
  int dsp, dct, dgrp, dtw, dth, dtd, dnb;

  __device__ __forceinline__ static void digits(const BoxTiling& t, uint32_t v, int& sp, int& ct,
                                                int& grp, int& tw, int& th, int& td, int& nb) {
    uint32_t q, r;
    fast_divmod(v, t.fd_split, q, r); sp = (int)r;
    fast_divmod(q, t.fd_ntiles, q, r); ct = (int)r;
    grp = (int)(q % (uint32_t)t.G); q /= (uint32_t)t.G;
    fast_divmod(q, t.fd_nTw, q, r); tw = (int)r;
    fast_divmod(q, t.fd_nTh, q, r); th = (int)r;
    fast_divmod(q, t.fd_nTd, q, r); td = (int)r;
    nb = (int)q;
  }
  __device__ __forceinline__ void init(const BoxTiling& t, long long first, long long step) {
    u = first;
    stride = step;
    digits(t, (uint32_t)(first < t.units ? first : 0), sp, ct, grp, tw, th, td, nb);
    digits(t, (uint32_t)(step < t.units ? step : t.units), dsp, dct, dgrp, dtw, dth, dtd, dnb);
  }
  __device__ __forceinline__ void next(const BoxTiling& t) {
    u += stride;
    int c;
    sp += dsp; c = sp >= t.split; if (c) sp -= t.split;
    ct += dct + c; c = ct >= t.ntiles; if (c) ct -= t.ntiles;
    grp += dgrp + c; c = grp >= t.G; if (c) grp -= t.G;
    tw += dtw + c; c = tw >= t.nTw; if (c) tw -= t.nTw;
    th += dth + c; c = th >= t.nTh; if (c) th -= t.nTh;
    td += dtd + c; c = td >= t.nTd; if (c) td -= t.nTd;
    nb += dnb + c;
  }
  __device__ __forceinline__ BoxUnit unit(const BoxTiling& t) const {
    BoxUnit b;
    b.n0 = nb * t.Nb;
    b.od0 = td * t.Dt;
    b.oh0 = th * t.Ht;
    b.ow0 = tw * t.Wt;
    b.grp = grp;
    b.ct = ct;
    b.sp = sp;
    b.c_begin = sp * t.chunks_per_split;
    b.nk = min(t.chunks_per_split, t.chunks - b.c_begin);
    return b;
  }
};

// Host: the box of output pixels for a geometry, the widest first (Wt up to max_wt), then
// rows (up to max_ht), depth slices (up to max_dt) and, when a box holds whole images,
// several images.
struct BoxShape {
  int Nb, Dt, Ht, Wt, rows, vec;
  long long boxes;
};

inline int imin(int a, int b) { return a < b ? a : b; }

// Rows and slices are spread evenly over the boxes (no nearly empty last box).
inline BoxShape box_shape(const ConvGeom& g, int max_px, int max_wt, int max_ht, int max_dt) {
  BoxShape t{};
  t.Wt = imin(imin(g.OW, max_wt), max_px);
  if (t.Wt < 1) t.Wt = 1;
  t.Ht = imin(imin(g.OH, max_ht), max_px / t.Wt);
  if (t.Ht < 1) t.Ht = 1;
  t.Ht = (g.OH + (g.OH + t.Ht - 1) / t.Ht - 1) / ((g.OH + t.Ht - 1) / t.Ht);
  // boxes of whole rows: an even count of 8-pixel runs per box when one more row allows it
  if (t.Wt == g.OW && t.Ht < g.OH && (t.Ht * g.OW) % 8 != 0) {
    for (int h = t.Ht + 1; h <= imin(imin(g.OH, max_ht), max_px / t.Wt); ++h)
      if ((h * g.OW) % 8 == 0) {
        t.Ht = h;
        break;
      }
  }
  t.Dt = imin(imin(g.OD, max_dt), max_px / (t.Wt * t.Ht));
  if (t.Dt < 1) t.Dt = 1;
  t.Dt = (g.OD + (g.OD + t.Dt - 1) / t.Dt - 1) / ((g.OD + t.Dt - 1) / t.Dt);
  const bool whole = t.Wt == g.OW && t.Ht == g.OH && t.Dt == g.OD;
  const int per = t.Wt * t.Ht * t.Dt;
  t.Nb = whole ? imin(g.N, max_px / per) : 1;
  if (t.Nb > 1) t.Nb = (g.N + (g.N + t.Nb - 1) / t.Nb - 1) / ((g.N + t.Nb - 1) / t.Nb);
  t.rows = t.Nb * t.Dt * t.Ht * t.Wt;
  t.boxes = (long long)((g.N + t.Nb - 1) / t.Nb) * ((g.OD + t.Dt - 1) / t.Dt) *
            ((g.OH + t.Ht - 1) / t.Ht) * ((g.OW + t.Wt - 1) / t.Wt);
  // 16-byte Y/Z vectors need every 8-pixel group of a box to be 8 consecutive, 16-byte
  // aligned pixels of one image: whole images, boxes of whole 8-pixel runs of a row, or
  // boxes of whole rows (one depth slice, or whole planes) whose pixel counts are multiples
  // of 8 (then every box starts 16-byte aligned and its pixels are consecutive in Y)
  const bool rows_run = t.Wt % 8 == 0 && g.OW % t.Wt == 0;
  const bool full_rows = t.Wt == g.OW && (t.Dt == 1 || t.Ht == g.OH) &&
                         (t.Dt * t.Ht * g.OW) % 8 == 0 && ((long long)g.OH * g.OW) % 8 == 0;
  t.vec = (g.P % 8 == 0) && (rows_run || full_rows || whole);
  return t;
}

inline BoxTiling make_box_tiling(const ConvGeom& g, const BoxShape& sh, int split, int chunks,
                                 int R = 1, int npx = kMaxPx) {
  BoxTiling t{};
  t.R = R;
  t.Mp = kMT / R;
  t.npx = npx;
  t.G = g.G;
  t.Nb = sh.Nb; t.Dt = sh.Dt; t.Ht = sh.Ht; t.Wt = sh.Wt;
  t.rows = sh.rows;
  t.vec = sh.vec;
  t.nTd = (g.OD + sh.Dt - 1) / sh.Dt;
  t.nTh = (g.OH + sh.Ht - 1) / sh.Ht;
  t.nTw = (g.OW + sh.Wt - 1) / sh.Wt;
  t.ntiles = (g.Mg + kMT - 1) / kMT;
  t.split = split;
  t.chunks = chunks;
  t.chunks_per_split = (chunks + split - 1) / split;
  t.units = sh.boxes * g.G * t.ntiles * split;
  t.fd_split = make_fastdiv((uint32_t)split);
  t.fd_gnt = make_fastdiv((uint32_t)(g.G * t.ntiles));
  t.fd_ntiles = make_fastdiv((uint32_t)t.ntiles);
  t.fd_nTw = make_fastdiv((uint32_t)t.nTw);
  t.fd_nTh = make_fastdiv((uint32_t)t.nTh);
  t.fd_nTd = make_fastdiv((uint32_t)t.nTd);
  return t;
}

// ------------------------------------------------------------------ epilogue

// Per-pixel entries of the box in shared memory, built once per CTA: {offset of the pixel in
// Y relative to the box origin (n0, od0, oh0, ow0) for channel 0, wt, ht, nb << 16 | dt}.
// Pixels past the box's rows get a wt that no box origin keeps inside Y.
__device__ __forceinline__ void build_pixel_table(const ConvGeom& g, const BoxTiling& t, int4* pix,
                                                  int npx) {
  for (int i = threadIdx.x; i < npx; i += blockDim.x) {
    int4 e = make_int4(0, 1 << 30, 0, 0);
    if (i < t.rows) {
      const int wt = i % t.Wt, ht = (i / t.Wt) % t.Ht, dt = (i / (t.Wt * t.Ht)) % t.Dt;
      const int nb = i / (t.Wt * t.Ht * t.Dt);
      const long long rel = (long long)nb * g.M * g.P + ((long long)dt * g.OH + ht) * g.OW + wt;
      e = make_int4((int)rel, wt, ht, (nb << 16) | dt);
    }
    pix[i] = e;
  }
}

__device__ __forceinline__ bool pixel_in(const ConvGeom& g, const BoxUnit& un, int4 e) {
  return un.ow0 + e.y < g.OW && un.oh0 + e.z < g.OH && un.od0 + (e.w & 0xffff) < g.OD &&
         un.n0 + (e.w >> 16) < g.N;
}

// Eight results rounded to f16 and packed for one 16-byte store.
template <int ACT>
__device__ __forceinline__ uint4 act_pack8(const float* v, float alpha, float beta) {
  uint32_t w[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const __half2 h = __floats2half2_rn(act_eval<ACT, true>(v[2 * j], alpha, beta),
                                        act_eval<ACT, true>(v[2 * j + 1], alpha, beta));
    w[j] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ void add_half8(float* v, uint4 z) {
  const uint32_t w[4] = {z.x, z.y, z.z, z.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const __half2 h = *reinterpret_cast<const __half2*>(&w[j]);
    v[2 * j] += __low2float(h);
    v[2 * j + 1] += __high2float(h);
  }
}

// Per-warp transpose tile of the epilogue: 32 channels x 64 pixels of f16, rows padded to
// 144 bytes so that both the row-wise 16-byte writes of the channel owners and the
// run-wise 16-byte reads of the storing lanes are free of bank conflicts.
constexpr uint32_t kTpPitch = 144;
constexpr uint32_t kTpBytes = 32 * kTpPitch;

// The epilogue warps of a box-tiled kernel (channel-major accumulator). Warp e: lane quarter
// e % 4 (channels 32 (e % 4) .. + 31 of the tile), set (e / 4) % SETS (takes the CTA's tiles
// tcount = set, set + SETS, ...), and the 64-pixel slabs (e / (4 SETS)) + WPQ k of the tile.
// Accumulator buffer of tile tcount: tcount % NACC, NPX columns wide. bias_s: the bias
// widened to f32 in shared memory, or null to read b. tp: this warp's transpose tile.
// Per slab, in the vector path (8-pixel runs of Y):
//   1. with Z: lane l loads Z of runs l % 8 for channel rows l / 8 + 4 i (coalesced 128-byte
//      runs of one channel) into the tile;
//   2. the channel owners (thread = channel) read 16 pixels per tcgen05.ld, add B and Z,
//      apply the activation, round to f16 and write their row of the tile;
//   3. lanes read the tile back the same way as in 1 and store Y as 16-byte vectors.
// Otherwise each owner stores its pixels one by one. With ACT == kActPartial the raw sums go
// to the f32 partials of the unit's split, 8 pixels per owner and store.
template <int NPX, int ACT, int NACC, int SETS, int WPQ>
__device__ __forceinline__ void box_epilogue(const ConvGeom& g, const BoxTiling& t,
                                             const __half* b, const float* bias_s,
                                             const __half* z, __half* y, float* part,
                                             uint64_t* acc_full, uint64_t* acc_empty,
                                             volatile int* abort_flag, uint32_t tmem,
                                             const int4* pix, uint32_t tp, int e, int lane) {
  static_assert((NACC & (NACC - 1)) == 0, "accumulator count is a power of two");
  const int q4 = e & 3;
  const int j = e >> 2;
  const int eset = j % SETS;
  const int s_first = (j / SETS) * 64;
  constexpr int kSlabStep = WPQ * 64;
  const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
  const long long MP = (long long)g.M * g.P;
  const bool vec = t.vec != 0;
  const bool hz = z != nullptr;
  const int rj = lane & 7;    // in phases 1 and 3: this lane's 8-pixel run of the slab
  const int rrow = lane >> 3; // ... and its first channel row (then + 4, + 8, ...)
  uint32_t tcount = (uint32_t)eset;
  UnitIter it;
  it.init(t, blockIdx.x + (long long)eset * gridDim.x, (long long)SETS * gridDim.x);
  for (; it.u < t.units; it.next(t), tcount += SETS) {
    if (*abort_flag) break;
    const BoxUnit un = it.unit(t);
    const uint32_t buf = tcount & (uint32_t)(NACC - 1);
    // this quarter's lanes hold band r = 32 q4 / Mp: channels of sub-box r (pixels r * npx ..)
    const int band = (q4 * 32) / t.Mp;
    const int c_tile = un.ct * kMT + (q4 * 32) % t.Mp;  // first channel of the quarter
    const int nrows = min(min(32, t.Mp), g.Mg - c_tile);  // valid channels (may be <= 0)
    const int m0 = un.grp * g.Mg + c_tile;                // output channel of row 0
    const int px0 = band * t.npx;                          // the sub-box's first box pixel
    const int prow = min(t.npx, t.rows - px0);             // the sub-box's pixels
    const bool m_ok = lane < nrows;
    const long long origin = (long long)un.n0 * MP + ((long long)un.od0 * g.OH + un.oh0) * g.OW + un.ow0;
    float bm = 0.0f;
    if (ACT != kActPartial && b && m_ok) bm = bias_s ? bias_s[m0 + lane] : __half2float(b[m0 + lane]);
    if (!bounded_wait(ptx::smem_addr(&acc_full[buf]), (tcount / (uint32_t)NACC) & 1u, abort_flag)) break;
    ptx::tc_fence_after();
    const uint32_t acc = lane_base + buf * (uint32_t)NPX;
    if (nrows > 0 && prow > 0) {
#pragma unroll 1
      for (int s = s_first; s < prow; s += kSlabStep) {
        if (ACT == kActPartial || !vec) {
          // the owners store their own pixels (split-K partials, or runs that are not 16-byte
          // vectors of Y)
          const long long chan = origin + (long long)(m_ok ? m0 + lane : 0) * g.P;
          float* pout = part + (long long)un.sp * g.N * MP;
#pragma unroll 1
          for (int c = s; c < s + 64 && c < prow; c += 8) {
            float v[8];
            ptx::tmem_ld8(acc + (uint32_t)c, v);
            if (!m_ok) continue;
            if (ACT == kActPartial && vec) {
              const int4 pe = pix[px0 + c];
              if (pixel_in(g, un, pe)) {
                float* pp = pout + chan + pe.x;
                ptx::st_global_v4(pp, make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]),
                                                 __float_as_uint(v[2]), __float_as_uint(v[3])));
                ptx::st_global_v4(pp + 4, make_uint4(__float_as_uint(v[4]), __float_as_uint(v[5]),
                                                     __float_as_uint(v[6]), __float_as_uint(v[7])));
              }
              continue;
            }
#pragma unroll 1
            for (int jj = 0; jj < 8; ++jj) {
              const int i = c + jj;
              if (i >= prow) break;
              const int4 pe = pix[px0 + i];
              if (!pixel_in(g, un, pe)) continue;
              const long long off = chan + pe.x;
              if constexpr (ACT == kActPartial) {
                pout[off] = v[jj];
              } else {
                float vv = v[jj] + bm;
                if (hz) vv += __half2float(z[off]);
                y[off] = __float2half_rn(act_eval<ACT, true>(vv, g.alpha, g.beta));
              }
            }
          }
          continue;
        }
        if constexpr (ACT != kActPartial) {
          // this lane's run of the slab in phases 1 and 3: its place in Y for channel row 0
          const int col = s + 8 * rj;
          bool run_ok = false;
          long long roff = 0;
          if (col < prow) {
            const int4 pe = pix[px0 + col];
            run_ok = pixel_in(g, un, pe);
            roff = origin + (long long)m0 * g.P + pe.x;
          }
          if (hz) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int row = rrow + 4 * i;
              uint4 zv = make_uint4(0, 0, 0, 0);
              if (run_ok && row < nrows) zv = ptx::ldg_nc_v4(z + roff + (long long)row * g.P);
              ptx::st_shared_v4(tp + (uint32_t)row * kTpPitch + 16u * (uint32_t)rj, zv.x, zv.y, zv.z, zv.w);
            }
            __syncwarp();
          }
          const uint32_t own = tp + (uint32_t)lane * kTpPitch;
#pragma unroll 1
          for (int gq = 0; gq < 4; ++gq) {
            const int c = s + 16 * gq;
            if (c >= prow) break;
            float v[16];
            ptx::tmem_ld16(acc + (uint32_t)c, v);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              float* vh = v + 8 * h;
              const uint32_t at = own + 32u * (uint32_t)gq + 16u * (uint32_t)h;
#pragma unroll
              for (int jj = 0; jj < 8; ++jj) vh[jj] += bm;
              if (hz) add_half8(vh, ptx::ld_shared_v4(at));
              const uint4 o = act_pack8<ACT>(vh, g.alpha, g.beta);
              ptx::st_shared_v4(at, o.x, o.y, o.z, o.w);
            }
          }
          __syncwarp();
          if (run_ok) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int row = rrow + 4 * i;
              if (row < nrows) {
                const uint4 o = ptx::ld_shared_v4(tp + (uint32_t)row * kTpPitch + 16u * (uint32_t)rj);
                ptx::st_global_v4(y + roff + (long long)row * g.P, o);
              }
            }
          }
          __syncwarp();
        }
      }
    }
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&acc_empty[buf]));
  }
}

// The bias widened to f32 into shared memory (all threads of the CTA; the caller
// synchronises before the epilogue reads it).
constexpr int kMaxSmemBias = 2048;  // output channels whose bias is staged
__device__ __forceinline__ void stage_bias(const __half* b, float* bs, int M) {
  for (int m = threadIdx.x; m < M; m += blockDim.x) bs[m] = __half2float(b[m]);
}

// Read and clear this translation unit's device error word (after synchronising `s`).
inline int read_and_clear_tc_error(cudaStream_t s, unsigned* value) {
  unsigned v = 0;
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return (int)e;
  e = cudaMemcpyFromSymbol(&v, g_tc_error, sizeof(v));
  if (e != cudaSuccess) return (int)e;
  if (v) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_tc_error, &zero, sizeof(zero));
    if (e != cudaSuccess) return (int)e;
  }
  *value = v;
  return 0;
}

}  // namespace
}  // namespace fconv
