// Implicit-GEMM FusedConv on tcgen05 with the im2col operand built in shared memory from the
// input patch of each tile (README variants implicit_im2col_tiled_reg: im2col elements are
// gathered straight from X into the GEMM tiles, "avoiding a materialized column scratch
// buffer"). X is read in its own NC(D)HW layout: nothing is repacked and no workspace is
// needed unless K is split.
//
// A tile is a box of at most 256 output pixels (tc_common.cuh) and 128 output channels; the
// accumulator is channel-major (TMEM lane = channel, column = pixel). For a block of Cb input
// channels the box's receptive field in X is a box too, the patch: PW x PH x PD positions
// (the x start rounded down to a multiple of 8 elements, as a TMA box requires) x Cb channels
// x Nb images. One 5-D TMA load brings the patch into shared memory and fills positions
// outside X with zeros, which is the convolution's zero padding. The GEMM's K runs in W's own
// order, k = c * KV + tap, so that the weights are read as they are:
//   A[pixel, k] = patch[pixel base + table[k']]       (k' = k - block * Cb * KV)
// where a pixel's base is its place in the patch and table[k'] the offset of channel c' and
// tap (kz, ky, kx) (dilation included). Each chunk is 64 consecutive k' of one block.
//
// Warps (one persistent CTA per SM):
//   0-7    epilogue: two sets of four (one warp per TMEM lane quarter of the tile's
//          channels) take the tiles in turn; 16 pixels per thread and tcgen05.ld, stored
//          through a per-warp transpose tile as coalesced runs (tc_common.cuh box_epilogue)
//   8-15   im2col builders: thread t writes row t (one output pixel) of the chunk's
//          128-byte-swizzled K-major tile from the patch (one shared-memory load per element,
//          one 16-byte store per 8 elements)
//   16     TMEM allocation and MMA issue (tcgen05.mma.cta_group::1.kind::f16, M = 128
//          channels, N = the box's pixels rounded up to 16)
//   17     TMA producer: the patches and, unless the weights are resident, the weight tiles
// Weights: when all of W fits (in GEMM order, zero padded to whole 128-channel tiles) in at
// most 48 KB it is copied into shared memory once per CTA (resident), so no weight tile moves
// per chunk; otherwise a 2-D TMA box of W (or of a copy with rows padded to a multiple of 8
// elements when W's row length is not) lands beside each im2col chunk.
// Convs with at most 64 output channels per group stack R = 128 / Mp sub-boxes of pixels in
// the accumulator's lanes (Mp = 64 or 32): the weights operand of sub-box r is a 128-row tile
// whose band r (rows r Mp ..) holds W and whose other rows are zero, and each chunk issues R
// MMAs into the same accumulator, so that every TMEM lane quarter carries channels and all
// four SM sub-partitions share the epilogue.
// When X's rows are not a multiple of 8 elements (TMA strides are multiples of 16 bytes),
// the builder warps load the patch themselves with plain loads (one patch slot, handed over
// through the same time-bounded mbarriers).
#include "tc_common.cuh"

#include <climits>
#include <cstring>

namespace fconv {
namespace {

constexpr int kPWarps = 18;
constexpr int kPThreads = kPWarps * 32;
constexpr int kPEpiWarps = 8;
constexpr int kPBuildWarp0 = 8;
constexpr int kPBuildWarps = 8;
constexpr int kPBuildThreads = kPBuildWarps * 32;  // one per pixel row, up to 256
constexpr int kPMmaWarp = 16;
constexpr int kPLoadWarp = 17;
constexpr int kMaxSlots = 8;               // patch slots (TMA loads in flight)
constexpr int kMaxTab = 1024;              // entries of the (channel, tap) offset table
constexpr uint32_t kResidentMax = 48 * 1024;
constexpr size_t kSmemBudget = 220 * 1024; // dynamic shared memory of one CTA

struct PatchArgs {
  BoxTiling t;
  const uint16_t* x;
  const uint16_t* w;       // W as given (read when the weights are resident)
  const __half* b;
  const __half* z;
  __half* y;
  float* part;             // split-K partials [split][N][M][P] (f32), or null
  int stages;
  uint32_t stage_bytes;    // weights chunk (unless resident) + im2col chunk
  uint32_t idesc;          // MMA instruction descriptor (M = 128, N = pixels rounded to 16)
  int Cb, nblk, cpb;       // channels per patch block, blocks per group, chunks per full block
  int Kb_full, Kb_last;    // K of a full block (Cb * KV) and of the group's last block
  int last_chunks;         // chunks of the group's last block
  int PW, PH, PD, plane;   // patch extents (PW a multiple of 8), plane = PD * PH * PW
  uint32_t slot_bytes;     // shared memory of one patch (1024-byte multiple)
  uint32_t patch_tx;       // bytes one TMA patch load delivers
  int nslot;
  int tma_x;               // patches by TMA (1) or by the builder warps' plain loads (0)
  int resident;            // weights resident in shared memory
  int mpad;                // resident weights: rows per group (ntiles * 128)
  uint32_t res_bytes;
  int R, Mp;               // stacked sub-boxes and the lanes of each (Mp = 128 / R)
  int pairs;               // taps (kx, kx+1) are adjacent, 4-byte aligned halves: 32-bit gathers
};

struct PatchCtl {
  uint64_t a_full[kMaxStages];   // im2col chunk built (the eight builder warps)
  uint64_t b_full[kMaxStages];   // weights chunk landed (TMA)
  uint64_t empty[kMaxStages];    // the MMAs reading the stage are done
  uint64_t p_full[kMaxSlots];
  uint64_t p_empty[kMaxSlots];
  uint64_t acc_full[kMaxAcc];
  uint64_t acc_empty[kMaxAcc];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

// Chunk q of a group's K: block q / cpb, first k' = 64 (q % cpb) of that block, valid length.
__device__ __forceinline__ void chunk_of(int q, const PatchArgs& a, int& blk, int& kin, int& len) {
  blk = q / a.cpb;
  kin = (q - blk * a.cpb) * kBK;
  const int kb = blk == a.nblk - 1 ? a.Kb_last : a.Kb_full;
  len = min(kBK, kb - kin);
}

__device__ __forceinline__ int floor8(int v) { return v & ~7; }

// The CTA's copy of the weights: for chunk q, group grp and row ml < mpad, the 128-byte
// swizzled K-major row ((q * G + grp) * mpad + ml) holds W[grp * Mg + ml][block k .. + 63],
// zero past the chunk's length and for rows past Mg. Loads of four 16-byte units are issued
// before any of them is stored.
// With stacked sub-boxes, tile ((q * G + grp) * ntiles + ct) * R + r of 128 rows holds W in
// its band r (rows r Mp .. r Mp + Mg - 1) and zeros elsewhere.
__device__ void load_resident_weights(const ConvGeom& g, const PatchArgs& a, uint32_t dst) {
  const int ntiles = a.mpad / kMT;
  const int rows = a.t.chunks * g.G * ntiles * a.R * kMT;
  for (int v0 = threadIdx.x; v0 < rows * 8; v0 += 4 * blockDim.x) {
    uint32_t e[4][8];
    uint32_t at[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const int v = v0 + h * blockDim.x;
      const int row = v >> 3, u = v & 7;
      const int T = row / kMT, mt = row - T * kMT;  // tile and its row
      const int r = T % a.R, T1 = T / a.R;
      const int ct = T1 % ntiles, T2 = T1 / ntiles;
      const int grp = T2 % g.G, q = T2 / g.G;
      const int ch = ct * kMT + (a.R > 1 ? mt - r * a.Mp : mt);  // channel within the group
      const bool in_band = a.R == 1 || (mt >= r * a.Mp && mt < (r + 1) * a.Mp);
      int blk, kin, len;
      chunk_of(q, a, blk, kin, len);
      at[h] = dst + (uint32_t)row * 128u + ((uint32_t)(u ^ (row & 7)) << 4);
      const bool ok = v < rows * 8 && in_band && ch < g.Mg;
      const uint16_t* src = a.w + (long long)(grp * g.Mg + (ok ? ch : 0)) * g.Kg + blk * a.Kb_full + kin;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int kk = 8 * u + j;
        e[h][j] = (ok && kk < len) ? (uint32_t)src[kk] : 0u;
      }
    }
#pragma unroll
    for (int h = 0; h < 4; ++h)
      if (v0 + h * (int)blockDim.x < rows * 8)
        ptx::st_shared_v4(at[h], e[h][0] | (e[h][1] << 16), e[h][2] | (e[h][3] << 16),
                          e[h][4] | (e[h][5] << 16), e[h][6] | (e[h][7] << 16));
  }
}

// Plain-load patch (builder warps, 256 threads): block blk of unit un into slot 0.
__device__ void load_patch_plain(const ConvGeom& g, const PatchArgs& a, const BoxUnit& un, int blk,
                                 uint16_t* ps, int btid) {
  const int xs = floor8(un.ow0 * g.sW - g.pW), ys = un.oh0 * g.sH - g.pH, zs = un.od0 * g.sD - g.pD;
  const int c0 = un.grp * g.Cg + blk * a.Cb;
  const int total = a.t.Nb * a.Cb * a.plane;
  for (int e = btid; e < total; e += kPBuildThreads) {
    int t = e;
    const int px = t % a.PW; t /= a.PW;
    const int py = t % a.PH; t /= a.PH;
    const int pz = t % a.PD; t /= a.PD;
    const int cc = t % a.Cb;
    const int nb = t / a.Cb;
    const int ix = xs + px, iy = ys + py, iz = zs + pz, c = c0 + cc, n = un.n0 + nb;
    uint16_t v = 0;
    if (ix >= 0 && ix < g.IW && iy >= 0 && iy < g.IH && iz >= 0 && iz < g.ID && c < g.C && n < g.N)
      v = a.x[(((long long)n * g.C + c) * g.ID + iz) * g.IH * (long long)g.IW + (long long)iy * g.IW + ix];
    ps[e] = v;
  }
}

template <int NPX, bool SPLIT>
__global__ void __launch_bounds__(kPThreads, 1)
    igemm_patch_kernel(const ConvGeom g, const PatchArgs a, const __grid_constant__ CUtensorMap tmap_x,
                       const __grid_constant__ CUtensorMap tmap_w) {
  using AP = AccPlan<NPX, kPEpiWarps>;

  extern __shared__ uint8_t dsmem[];
  __shared__ PatchCtl ctl;
  __shared__ __align__(16) int tab[kMaxTab];

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t base = (ptx::smem_addr(dsmem) + 1023u) & ~1023u;
  uint8_t* gbase = dsmem + (base - ptx::smem_addr(dsmem));
  const int S = a.stages;
  // each stage: [R weights tiles of 16 KB unless resident][R im2col tiles of NPX x 128 B]
  const uint32_t wst = a.resident ? 0u : (uint32_t)a.R * kWBytes;  // im2col tiles' offset
  const uint32_t res_off = (uint32_t)S * a.stage_bytes;
  const uint32_t p_off = res_off + a.res_bytes;
  const uint32_t pix_off = p_off + (uint32_t)a.nslot * a.slot_bytes;
  const uint32_t bias_off = pix_off + (uint32_t)(a.R * NPX) * 16;
  const uint32_t tp_off = bias_off + kMaxSmemBias * 4;  // the epilogue warps' transpose tiles

  // byte offset of (channel c', tap) from a pixel's base in the patch, for k' = c' * KV + tap
  for (int k = tid; k < kMaxTab; k += kPThreads) {
    int v = 0;
    if (k < a.Kb_full) {
      const int c = k / g.KV, tap = k - c * g.KV;
      const int kx = tap % g.KW, ky = (tap / g.KW) % g.KH, kz = tap / (g.KW * g.KH);
      v = 2 * (c * a.plane + (kz * g.dD * a.PH + ky * g.dH) * a.PW + kx * g.dW);
    }
    tab[k] = v;
  }
  int4* pix = reinterpret_cast<int4*>(gbase + pix_off);
  build_pixel_table(g, a.t, pix, a.R * NPX);
  if (!a.resident && a.R > 1) {
    // the weights tiles' rows outside their band stay zero (TMA writes only the band)
    for (int s = 0; s < S; ++s)
      for (uint32_t o = (uint32_t)tid * 16u; o < (uint32_t)a.R * kWBytes; o += kPThreads * 16u)
        ptx::st_shared_v4(base + (uint32_t)s * a.stage_bytes + o, 0u, 0u, 0u, 0u);
    ptx::fence_proxy_async_smem();
  }
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(ptx::smem_addr(&ctl.a_full[s]), kPBuildWarps);
      ptx::mbar_init(ptx::smem_addr(&ctl.b_full[s]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl.empty[s]), 1);
    }
    for (int s = 0; s < kMaxSlots; ++s) {
      // a TMA patch completes on the producer's arrival and its bytes; a plain-load patch
      // on the arrivals of the eight builder warps that load it
      ptx::mbar_init(ptx::smem_addr(&ctl.p_full[s]), a.tma_x ? 1 : kPBuildWarps);
      ptx::mbar_init(ptx::smem_addr(&ctl.p_empty[s]), kPBuildWarps);
    }
    for (int b = 0; b < AP::nacc; ++b) {
      ptx::mbar_init(ptx::smem_addr(&ctl.acc_full[b]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl.acc_empty[b]), kPEpiWarps / AP::sets);
    }
    ptx::mbar_init(ptx::smem_addr(&ctl.drain), 1);
    ctl.abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kPMmaWarp) {
    ptx::tmem_alloc(ptx::smem_addr(&ctl.tmem_base), AP::tmem_cols);
    ptx::tmem_relinquish();
  }
  if (warp == kPLoadWarp && lane == 0) {
    if (a.tma_x) ptx::prefetch_tmap(&tmap_x);
    if (!a.resident) ptx::prefetch_tmap(&tmap_w);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  volatile int* abort_flag = &ctl.abort_flag;
  ptx::pdl_wait();  // X, W, B and Z may be the previous kernel's outputs
  float* bias_s = nullptr;  // bias widened to f32 (read by the epilogue warps)
  if (a.b && g.M <= kMaxSmemBias) {
    bias_s = reinterpret_cast<float*>(gbase + bias_off);
    stage_bias(a.b, bias_s, g.M);
  }
  if (a.resident) {
    load_resident_weights(g, a, base + res_off);
    ptx::fence_proxy_async_smem();  // the MMA reads them through the async proxy
  }
  __syncthreads();

  if (warp >= kPBuildWarp0 && warp < kPBuildWarp0 + kPBuildWarps) {
    // ================================================================ im2col builders
    // box pixels i0 and i0 + 256 (when R * NPX > 256): sub-box i / NPX, row i % NPX
    const int i = (warp - kPBuildWarp0) * 32 + lane;
    const int nrow = (a.R * NPX + kPBuildThreads - 1) / kPBuildThreads;
    // at most 128 rows a chunk: two threads per row, each writing half of its 16-byte units
    const bool halves = a.R * NPX <= kPBuildThreads / 2;
    const int ri = halves ? (i & (kPBuildThreads / 2 - 1)) : i;
    const int half = halves ? (i / (kPBuildThreads / 2)) : 0;
    int rbase[2] = {0, 0};
    uint32_t roff[2] = {0u, 0u};
    bool row_ok[2] = {false, false};
    // With stacked sub-boxes an im2col row past the box is not ignored: its column of the
    // accumulator holds the other bands' pixels, to which the band's MMA adds 0 x the row,
    // so the row must hold finite values (zeros); without stacking it is never read back.
    bool row_zero[2] = {false, false};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int pi = ri + h * kPBuildThreads;
      row_ok[h] = h < nrow && pi < a.t.rows;
      row_zero[h] = a.R > 1 && h < nrow && pi >= a.t.rows && pi < a.R * NPX;
      const int wt = pi % a.t.Wt, ht = (pi / a.t.Wt) % a.t.Ht, dt = (pi / (a.t.Wt * a.t.Ht)) % a.t.Dt;
      const int nb = pi / (a.t.Wt * a.t.Ht * a.t.Dt);
      // this pixel's place in the patch (elements), before the tile's x alignment offset
      rbase[h] = nb * a.Cb * a.plane + (dt * g.sD * a.PH + ht * g.sH) * a.PW + wt * g.sW;
      // its 128-byte row in the stage: im2col tile pi / NPX, row pi % NPX
      roff[h] = (uint32_t)(pi / NPX) * (uint32_t)(NPX * 128) + (uint32_t)(pi % NPX) * 128u;
    }
    Ring st{0, 0}, pr{0, 0};
    UnitIter it;
    it.init(a.t, blockIdx.x, gridDim.x);
    bool stop = false;
    for (; it.u < a.t.units && !stop; it.next(a.t)) {
      if (*abort_flag) break;
      const BoxUnit un = it.unit(a.t);
      const int xo = un.ow0 * g.sW - g.pW;
      const int ao = xo - floor8(xo);
      int blk = 0, i0 = 0;
      if (a.t.split > 1) {
        blk = un.c_begin / a.cpb;
        i0 = un.c_begin - blk * a.cpb;
      }
      for (int left = un.nk; left > 0 && !stop; ++blk, i0 = 0) {
        const int cin = blk == a.nblk - 1 ? a.last_chunks : a.cpb;  // chunks of this block
        const int n = min(left, cin - i0);
        if (!a.tma_x) {
          // one slot, filled by the eight builder warps together: wait until every builder
          // is done with the previous patch, load, then announce this warp's part
          if (!bounded_wait(ptx::smem_addr(&ctl.p_empty[0]), pr.phase ^ 1u, abort_flag)) {
            stop = true;
            break;
          }
          load_patch_plain(g, a, un, blk, reinterpret_cast<uint16_t*>(gbase + p_off), i);
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&ctl.p_full[0]));
        }
        if (!bounded_wait(ptx::smem_addr(&ctl.p_full[pr.idx]), pr.phase, abort_flag)) {
          stop = true;
          break;
        }
        const uint32_t pslot = base + p_off + pr.idx * a.slot_bytes;
        const int kb = blk == a.nblk - 1 ? a.Kb_last : a.Kb_full;
        for (int k = 0; k < n; ++k) {
          if (!bounded_wait(ptx::smem_addr(&ctl.empty[st.idx]), st.phase ^ 1u, abort_flag)) {
            stop = true;
            break;
          }
          const int kin = (i0 + k) * kBK;
          const int len = min(kBK, kb - kin);
          const int nunits = ((len + 15) >> 4) * 2;  // 16-byte units the MMAs read (even)
          // this thread's units of its rows: all, or one (even-aligned) half
          int u_lo = 0, u_hi = nunits;
          if (halves) {
            const int mid = ((nunits >> 1) + 1) & ~1;
            u_lo = half ? mid : 0;
            u_hi = half ? nunits : mid;
          }
          const uint32_t stg = base + st.idx * a.stage_bytes + wst;
#pragma unroll
          for (int h = 0; h < 2; ++h)
            if (row_zero[h])
              for (int uu = u_lo; uu < u_hi; ++uu)
                ptx::st_shared_v4(stg + roff[h] + (((uint32_t)uu ^ ((roff[h] >> 7) & 7u)) << 4), 0u, 0u, 0u, 0u);
          // two units per step, their table entries shared by this thread's rows: the loads
          // of both units and rows are independent and in flight together
          const int* tk = tab + kin;
          if (a.pairs) {
            // stride == kernel along x (even stride, even kernel width, dilation 1, even left
            // pad): the taps kx, kx + 1 of a pixel are neighbours in the patch and the pair
            // starts on a 4-byte boundary, so one 32-bit load brings two k values already in
            // the order the row wants (len is even: K per block is a multiple of KW)
#pragma unroll 1
            for (int uu = u_lo; uu < u_hi; uu += 2) {
              const int k0 = 8 * uu;
              const int4 t0 = *reinterpret_cast<const int4*>(tk + k0);
              const int4 t1 = *reinterpret_cast<const int4*>(tk + k0 + 4);
              const int4 t2 = *reinterpret_cast<const int4*>(tk + k0 + 8);
              const int4 t3 = *reinterpret_cast<const int4*>(tk + k0 + 12);
              const bool full = k0 + 16 <= len;
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                if (h >= nrow || !row_ok[h]) continue;
                const uint32_t src = pslot + 2u * (uint32_t)(rbase[h] + ao);
                auto ldp = [&](int off, int j) -> uint32_t {
                  return (full || k0 + 2 * j < len) ? ptx::ld_shared_u32(src + off) : 0u;
                };
                const uint32_t e0 = ldp(t0.x, 0), e1 = ldp(t0.z, 1), e2 = ldp(t1.x, 2), e3 = ldp(t1.z, 3);
                const uint32_t f0 = ldp(t2.x, 4), f1 = ldp(t2.z, 5), f2 = ldp(t3.x, 6), f3 = ldp(t3.z, 7);
                const uint32_t arow = stg + roff[h];
                const uint32_t swz = (roff[h] >> 7) & 7u;
                ptx::st_shared_v4(arow + (((uint32_t)uu ^ swz) << 4), e0, e1, e2, e3);
                ptx::st_shared_v4(arow + (((uint32_t)(uu + 1) ^ swz) << 4), f0, f1, f2, f3);
              }
            }
          } else
#pragma unroll 1
          for (int uu = u_lo; uu < u_hi; uu += 2) {
            const int k0 = 8 * uu;
            const int4 t0 = *reinterpret_cast<const int4*>(tk + k0);
            const int4 t1 = *reinterpret_cast<const int4*>(tk + k0 + 4);
            const int4 t2 = *reinterpret_cast<const int4*>(tk + k0 + 8);
            const int4 t3 = *reinterpret_cast<const int4*>(tk + k0 + 12);
            const bool full = k0 + 16 <= len;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              if (h >= nrow || !row_ok[h]) continue;
              const uint32_t src = pslot + 2u * (uint32_t)(rbase[h] + ao);
              auto ld = [&](int off, int j) -> uint32_t {
                return (full || k0 + j < len) ? ptx::ld_shared_u16(src + off) : 0u;
              };
              const uint32_t e0 = ld(t0.x, 0), e1 = ld(t0.y, 1), e2 = ld(t0.z, 2), e3 = ld(t0.w, 3);
              const uint32_t e4 = ld(t1.x, 4), e5 = ld(t1.y, 5), e6 = ld(t1.z, 6), e7 = ld(t1.w, 7);
              const uint32_t f0 = ld(t2.x, 8), f1 = ld(t2.y, 9), f2 = ld(t2.z, 10), f3 = ld(t2.w, 11);
              const uint32_t f4 = ld(t3.x, 12), f5 = ld(t3.y, 13), f6 = ld(t3.z, 14), f7 = ld(t3.w, 15);
              const uint32_t arow = stg + roff[h];
              const uint32_t swz = (roff[h] >> 7) & 7u;
              ptx::st_shared_v4(arow + (((uint32_t)uu ^ swz) << 4), e0 | (e1 << 16), e2 | (e3 << 16),
                                e4 | (e5 << 16), e6 | (e7 << 16));
              ptx::st_shared_v4(arow + (((uint32_t)(uu + 1) ^ swz) << 4), f0 | (f1 << 16),
                                f2 | (f3 << 16), f4 | (f5 << 16), f6 | (f7 << 16));
            }
          }
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&ctl.a_full[st.idx]));
          st.next((uint32_t)S);
        }
        if (stop) break;
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&ctl.p_empty[pr.idx]));
        pr.next((uint32_t)a.nslot);
        left -= n;
      }
    }
  } else if (warp == kPLoadWarp) {
    // ================================================================ TMA producer
    if (lane == 0) {
      Ring st{0, 0}, pr{0, 0};
      uint32_t armed_b = 0, armed_p = 0;
      UnitIter it;
      it.init(a.t, blockIdx.x, gridDim.x);
      bool stop = false;
      for (; it.u < a.t.units && !stop; it.next(a.t)) {
        if (*abort_flag) break;
        const BoxUnit un = it.unit(a.t);
        int blk = 0, i0 = 0;
        if (a.t.split > 1) {
          blk = un.c_begin / a.cpb;
          i0 = un.c_begin - blk * a.cpb;
        }
        for (int left = un.nk; left > 0 && !stop; ++blk, i0 = 0) {
          const int cin = blk == a.nblk - 1 ? a.last_chunks : a.cpb;
          const int n = min(left, cin - i0);
          if (a.tma_x) {
            if (!bounded_wait(ptx::smem_addr(&ctl.p_empty[pr.idx]), pr.phase ^ 1u, abort_flag)) {
              stop = true;
              break;
            }
            const uint32_t bar = ptx::smem_addr(&ctl.p_full[pr.idx]);
            ptx::mbar_arrive_expect_tx(bar, a.patch_tx);
            ptx::tma_load_5d(base + p_off + pr.idx * a.slot_bytes, &tmap_x,
                             floor8(un.ow0 * g.sW - g.pW), un.oh0 * g.sH - g.pH,
                             un.od0 * g.sD - g.pD, un.grp * g.Cg + blk * a.Cb, un.n0, bar);
            ++armed_p;
            pr.next((uint32_t)a.nslot);
          }
          if (!a.resident) {
            for (int k = 0; k < n; ++k) {
              if (!bounded_wait(ptx::smem_addr(&ctl.empty[st.idx]), st.phase ^ 1u, abort_flag)) {
                stop = true;
                break;
              }
              const uint32_t bar = ptx::smem_addr(&ctl.b_full[st.idx]);
              ptx::mbar_arrive_expect_tx(bar, (uint32_t)a.R * (uint32_t)a.Mp * 128u);
              for (int r = 0; r < a.R; ++r)  // band r of weights tile r
                ptx::tma_load_2d(base + st.idx * a.stage_bytes + (uint32_t)r * kWBytes +
                                     (uint32_t)(r * a.Mp) * 128u,
                                 &tmap_w, blk * a.Kb_full + (i0 + k) * kBK,
                                 un.grp * g.Mg + un.ct * kMT, bar);
              ++armed_b;
              st.next((uint32_t)S);
            }
          }
          left -= n;
        }
      }
      if (*abort_flag) {
        if (a.tma_x) drain_armed(ctl.p_full, armed_p, a.nslot);
        if (!a.resident) drain_armed(ctl.b_full, armed_b, S);
      }
    }
  } else if (warp == kPMmaWarp) {
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
        int blk = 0, i0 = 0;
        if (a.t.split > 1) {
          blk = un.c_begin / a.cpb;
          i0 = un.c_begin - blk * a.cpb;
        }
        for (int c = 0; c < un.nk; ++c) {
          if (!bounded_wait(ptx::smem_addr(&ctl.a_full[st.idx]), st.phase, abort_flag) ||
              (!a.resident && !bounded_wait(ptx::smem_addr(&ctl.b_full[st.idx]), st.phase, abort_flag))) {
            stop = true;
            break;
          }
          ptx::tc_fence_after();
          const int kb = blk == a.nblk - 1 ? a.Kb_last : a.Kb_full;
          const int len = min(kBK, kb - i0 * kBK);
          const uint32_t sbase = base + st.idx * a.stage_bytes;
          const uint32_t q = (uint32_t)(blk * a.cpb + i0);  // the group's chunk index
          const uint32_t wbase =
              a.resident ? base + res_off + (((q * (uint32_t)g.G + (uint32_t)un.grp) * (uint32_t)(a.mpad / kMT) +
                                              (uint32_t)un.ct) * (uint32_t)a.R) * kWBytes
                         : sbase;
          const uint32_t pbase = sbase + wst;
          const int ksteps = (len + 15) >> 4;
          for (int kk = 0; kk < ksteps; ++kk)
            for (int r = 0; r < a.R; ++r)
              ptx::mma_f16(dacc, ptx::desc_sw128(wbase + (uint32_t)r * kWBytes + kk * 32),
                           ptx::desc_sw128(pbase + (uint32_t)(r * NPX * 128) + kk * 32), a.idesc,
                           (c > 0 || kk > 0 || r > 0) ? 1u : 0u);
          ptx::mma_commit(ptx::smem_addr(&ctl.empty[st.idx]));
          st.next((uint32_t)S);
          if (++i0 == (blk == a.nblk - 1 ? a.last_chunks : a.cpb)) {
            ++blk;
            i0 = 0;
          }
        }
        if (stop) break;
        ptx::mma_commit(ptx::smem_addr(&ctl.acc_full[acc.idx]));
        acc.next((uint32_t)AP::nacc);
      }
      // every issued MMA must be complete before TMEM is freed
      ptx::mma_commit(ptx::smem_addr(&ctl.drain));
      drain_wait(ptx::smem_addr(&ctl.drain), 0);
    }
  } else if (warp < kPEpiWarps) {
    // ================================================================ epilogue (warps 0-15)
    // one loop per activation, chosen once: the group loop carries no dispatch
#define FCONV_EPI_LOOP(ACT)                                                                      \
  box_epilogue<NPX, ACT, AP::nacc, AP::sets, AP::wpq>(g, a.t, a.b, bias_s, a.z, a.y, a.part,     \
                                                     ctl.acc_full, ctl.acc_empty, abort_flag, tmem, \
                                                     pix, base + tp_off + (uint32_t)warp * kTpBytes, warp, lane)
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
  if (warp == kPMmaWarp) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, AP::tmem_cols);
  }
}

// W with rows padded to kpad (a multiple of 8) columns, for TMA boxes when W's own row
// length is not a multiple of 8 elements. One thread per 8 output columns.
__global__ void __launch_bounds__(256) pad_weights_kernel(const uint16_t* __restrict__ w,
                                                          uint16_t* __restrict__ wp, int M, int Kg,
                                                          int kpad) {
  ptx::pdl_wait();
  ptx::pdl_trigger();
  const long long units = (long long)M * (kpad / 8);
  for (long long v = blockIdx.x * 256LL + threadIdx.x; v < units; v += (long long)gridDim.x * 256) {
    const int m = (int)(v / (kpad / 8)), k0 = (int)(v - (long long)m * (kpad / 8)) * 8;
    uint32_t e[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) e[j] = k0 + j < Kg ? (uint32_t)w[(long long)m * Kg + k0 + j] : 0u;
    *reinterpret_cast<uint4*>(wp + (long long)m * kpad + k0) =
        make_uint4(e[0] | (e[1] << 16), e[2] | (e[3] << 16), e[4] | (e[5] << 16), e[6] | (e[7] << 16));
  }
}

// ------------------------------------------------------------------- host side

struct PatchPlan {
  bool ok;
  int npx;                 // pixel tile of the kernel instantiation (64, 128, 256)
  int R;                   // stacked sub-boxes (accumulator bands)
  BoxShape box;
  int Cb, nblk, cpb, Kb_full, Kb_last, chunks;
  int PW, PH, PD, plane;
  uint32_t slot_bytes, patch_tx, stage_bytes;
  int nslot, stages, tma_x, resident, mpad, pad_w, kpad;
  uint32_t res_bytes;
  size_t smem;
};

uint32_t round_up_u32(uint64_t v, uint64_t a) { return (uint32_t)((v + a - 1) / a * a); }

// Geometry of the patch for a box shape; false when the patch cannot be a TMA-sized box.
bool patch_extents(const ConvGeom& g, PatchPlan& p) {
  const BoxShape& b = p.box;
  // the largest x alignment offset over the boxes along a row
  int ao_max = 0;
  const int ntw = (g.OW + b.Wt - 1) / b.Wt;
  for (int i = 0; i < ntw && ao_max < 7; ++i) {
    const int xo = i * b.Wt * g.sW - g.pW;
    const int ao = xo - (xo & ~7);
    if (ao > ao_max) ao_max = ao;
  }
  p.PW = (ao_max + (b.Wt - 1) * g.sW + (g.KW - 1) * g.dW + 1 + 7) / 8 * 8;
  p.PH = (b.Ht - 1) * g.sH + (g.KH - 1) * g.dH + 1;
  p.PD = (b.Dt - 1) * g.sD + (g.KD - 1) * g.dD + 1;
  p.plane = p.PD * p.PH * p.PW;
  return p.PW <= 256 && p.PH <= 256 && p.PD <= 256 && b.Nb <= 256;
}

// The largest pixel tile (at most max_px) whose patches, operand ring and tables fit.
PatchPlan patch_plan(const ConvGeom& g, int max_px) {
  PatchPlan p{};
  p.ok = false;
  if (g.dtype != FCONV_F16) return p;
  // patch extents at most 256 per TMA box dimension
  const int wt_max = (256 - 8 - (g.KW - 1) * g.dW) / g.sW + 1;
  const int ht_max = (256 - 1 - (g.KH - 1) * g.dH) / g.sH + 1;
  const int dt_max = (256 - 1 - (g.KD - 1) * g.dD) / g.sD + 1;
  if (wt_max < 1 || ht_max < 1 || dt_max < 1) return p;
  // 32-bit indexing of units, pixel offsets and the table
  if ((long long)g.N * g.P * g.M >= 0x7fffffffLL) return p;
  // channels per block: all of C/group below 8, else a multiple of 8 (TMA boxes of the
  // weights start at multiples of 8 elements), at most what the table holds
  if (g.Cg < 8 && g.Cg * g.KV > kMaxTab) return p;
  if (g.Cg >= 8 && 8 * g.KV > kMaxTab) return p;
  const int cb_hi = g.Cg < 8 ? g.Cg : imin((g.Cg / 8) * 8, (kMaxTab / g.KV) / 8 * 8);
  p.tma_x = (g.IW % 8) == 0;
  const int ntiles = (g.Mg + kMT - 1) / kMT;
  p.mpad = ntiles * kMT;
  // as many stacked bands as the channels allow, fewer when they do not fit
  for (int R = g.Mg <= 32 ? 4 : g.Mg <= 64 ? 2 : 1; R >= 1; R /= 2)
  for (int px = kMaxPx; px >= 64; px /= 2) {
    p.R = R;
    if (px > max_px) continue;
    p.npx = px;
    p.box = box_shape(g, p.R * px, wt_max, ht_max, dt_max);
    if (p.box.rows > p.R * px || !patch_extents(g, p)) continue;
    // a smaller instantiation holds the box
    if (px > 64 && p.box.rows <= p.R * px / 2) continue;
    // blocks of C/group below 8: all of them, or (when a block's K stays a multiple of 8
    // elements, as the weight boxes need) fewer, down to one channel per patch
    for (int cb = cb_hi; cb >= 1; cb -= (g.Cg < 8 ? 1 : 8)) {
      if (g.Cg < 8 && cb != g.Cg && (cb * g.KV) % 8 != 0) continue;
      p.Cb = cb;
      p.nblk = (g.Cg + cb - 1) / cb;
      p.Kb_full = cb * g.KV;
      p.Kb_last = (g.Cg - (p.nblk - 1) * cb) * g.KV;
      p.cpb = (p.Kb_full + kBK - 1) / kBK;
      p.chunks = (p.nblk - 1) * p.cpb + (p.Kb_last + kBK - 1) / kBK;
      p.patch_tx = (uint32_t)((uint64_t)p.box.Nb * cb * p.plane * 2);
      p.slot_bytes = round_up_u32(p.patch_tx, 1024);
      const uint64_t res = (uint64_t)p.chunks * g.G * ntiles * p.R * kWBytes;
      p.resident = res <= kResidentMax ? 1 : 0;
      p.res_bytes = p.resident ? (uint32_t)res : 0;
      p.pad_w = (!p.resident && (g.Kg % 8) != 0) ? 1 : 0;
      p.kpad = p.pad_w ? (g.Kg + 7) / 8 * 8 : g.Kg;
      p.stage_bytes = (uint32_t)p.R * ((p.resident ? 0u : kWBytes) + (uint32_t)px * 128u);
      const size_t tables =
          (size_t)p.R * px * 16 + (size_t)kMaxSmemBias * 4 + kPEpiWarps * kTpBytes + 1024;
      for (int st = 4; st >= 2; --st) {
        const size_t fixed = (size_t)st * p.stage_bytes + p.res_bytes + tables;
        const int min_slots = p.tma_x ? 2 : 1;
        if (fixed + (size_t)min_slots * p.slot_bytes > kSmemBudget) continue;
        p.stages = st;
        p.nslot = min_slots;
        // more patches in flight while shared memory allows (TMA patches only)
        while (p.tma_x && p.nslot < kMaxSlots && fixed + (size_t)(p.nslot + 1) * p.slot_bytes <= kSmemBudget)
          ++p.nslot;
        p.smem = fixed + (size_t)p.nslot * p.slot_bytes;
        p.ok = true;
        return p;
      }
    }
  }
  return p;
}

template <int NPX, bool SPLIT>
int launch_patch_t(const ConvGeom& g, const IgemmConfig& c, const PatchArgs& pa, const CUtensorMap& tx,
                   const CUtensorMap& tw, size_t smem, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(igemm_patch_kernel<NPX, SPLIT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int)e;
  return launch_pdl(igemm_patch_kernel<NPX, SPLIT>, dim3((unsigned)c.grid), dim3(kPThreads), smem, s,
                    g, pa, tx, tw);
}

}  // namespace

bool igemm_patch_capable(const ConvGeom& g, int max_px) { return patch_plan(g, max_px).ok; }

long long igemm_patch_mtiles(const ConvGeom& g, int max_px) { return patch_plan(g, max_px).box.boxes; }

int igemm_patch_chunks(const ConvGeom& g, int max_px) { return patch_plan(g, max_px).chunks; }

size_t igemm_patch_workspace_bytes(const ConvGeom& g, const IgemmConfig& c) {
  const PatchPlan p = patch_plan(g, c.tile_n);
  size_t b = p.pad_w ? ((size_t)g.M * p.kpad * 2 + 1023) / 1024 * 1024 : 0;
  if (c.split_k > 1) b += (size_t)c.split_k * (size_t)g.N * (size_t)g.M * (size_t)g.P * 4;
  return b;
}

int igemm_patch_launches(const ConvGeom& g, const IgemmConfig& c) {
  const PatchPlan p = patch_plan(g, c.tile_n);
  return 1 + (p.pad_w ? 1 : 0) + (c.split_k > 1 ? 1 : 0);
}

int launch_igemm_patch(const ConvGeom& g, const IgemmConfig& c, const ConvArgs& a, void* stream) {
  cudaStream_t s = (cudaStream_t)stream;
  const PatchPlan p = patch_plan(g, c.tile_n);
  if (!p.ok) return (int)cudaErrorInvalidValue;
  EncodeTiledFn enc = tensor_map_encoder();
  if (!enc) return (int)cudaErrorNotSupported;
  uint8_t* ws = (uint8_t*)a.ws;
  const size_t wpad_bytes = p.pad_w ? ((size_t)g.M * p.kpad * 2 + 1023) / 1024 * 1024 : 0;
  if (p.pad_w) {
    long long blocks = ((long long)g.M * (p.kpad / 8) + 255) / 256;
    if (blocks > 152LL * 8) blocks = 152LL * 8;
    const int e = launch_pdl(pad_weights_kernel, dim3((unsigned)blocks), dim3(256), 0, s,
                             (const uint16_t*)a.w, (uint16_t*)ws, g.M, g.Kg, p.kpad);
    if (e != 0) return e;
  }
  CUtensorMap tx, tw;
  std::memset(&tx, 0, sizeof(tx));
  std::memset(&tw, 0, sizeof(tw));
  if (p.tma_x) {
    const cuuint64_t dims[5] = {(cuuint64_t)g.IW, (cuuint64_t)g.IH, (cuuint64_t)g.ID,
                                (cuuint64_t)g.C, (cuuint64_t)g.N};
    const cuuint64_t str[4] = {(cuuint64_t)g.IW * 2, (cuuint64_t)g.IH * g.IW * 2,
                               (cuuint64_t)g.IS * 2, (cuuint64_t)g.C * g.IS * 2};
    const cuuint32_t box[5] = {(cuuint32_t)p.PW, (cuuint32_t)p.PH, (cuuint32_t)p.PD,
                               (cuuint32_t)p.Cb, (cuuint32_t)p.box.Nb};
    const cuuint32_t es[5] = {1, 1, 1, 1, 1};
    const CUresult cr = enc(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 5, (void*)a.x, dims, str, box, es,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS) return (int)cudaErrorInvalidValue;
  }
  if (!p.resident) {
    const void* wmat = p.pad_w ? (const void*)ws : a.w;
    const cuuint64_t dims[2] = {(cuuint64_t)p.kpad, (cuuint64_t)g.M};
    const cuuint64_t str[1] = {(cuuint64_t)p.kpad * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)(kMT / p.R)};  // one band
    const cuuint32_t es[2] = {1, 1};
    const CUresult cr = enc(&tw, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, (void*)wmat, dims, str, box, es,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS) return (int)cudaErrorInvalidValue;
  }
  PatchArgs pa{};
  pa.t = make_box_tiling(g, p.box, c.split_k, p.chunks, p.R, p.npx);
  pa.x = (const uint16_t*)a.x;
  pa.w = (const uint16_t*)a.w;
  pa.b = (const __half*)a.b;
  pa.z = (const __half*)a.z;
  pa.y = (__half*)a.y;
  pa.part = c.split_k > 1 ? (float*)(ws + wpad_bytes) : nullptr;
  pa.stages = p.stages;
  pa.stage_bytes = p.stage_bytes;
  pa.idesc = ptx::idesc_f16_f32(kMT, p.R > 1 ? p.npx : (p.box.rows + 15) / 16 * 16);
  pa.Cb = p.Cb; pa.nblk = p.nblk; pa.cpb = p.cpb;
  pa.Kb_full = p.Kb_full; pa.Kb_last = p.Kb_last;
  pa.last_chunks = (p.Kb_last + kBK - 1) / kBK;
  pa.PW = p.PW; pa.PH = p.PH; pa.PD = p.PD; pa.plane = p.plane;
  pa.slot_bytes = p.slot_bytes;
  pa.patch_tx = p.patch_tx;
  pa.nslot = p.nslot;
  pa.tma_x = p.tma_x;
  pa.resident = p.resident;
  pa.mpad = p.mpad;
  pa.res_bytes = p.res_bytes;
  pa.R = p.R;
  pa.pairs = (g.sW % 2 == 0 && g.KW % 2 == 0 && g.dW == 1 && g.pW % 2 == 0) ? 1 : 0;
  pa.Mp = kMT / p.R;
  const bool sp = c.split_k > 1;
  int err;
  switch (p.npx) {
#define FCONV_PATCH_NPX(NPX)                                                                   \
  case NPX:                                                                                    \
    err = sp ? launch_patch_t<NPX, true>(g, c, pa, tx, tw, p.smem, s)                          \
             : launch_patch_t<NPX, false>(g, c, pa, tx, tw, p.smem, s);                        \
    break;
    FCONV_PATCH_NPX(64)
    FCONV_PATCH_NPX(128)
    FCONV_PATCH_NPX(256)
#undef FCONV_PATCH_NPX
    default: return (int)cudaErrorInvalidValue;
  }
  if (err != 0 || !sp) return err;
  return launch_splitk_reduce(g, c.split_k, pa.part, a.b, a.z, a.y, stream);
}

int read_and_clear_patch_error(void* stream, unsigned* value) {
  return read_and_clear_tc_error((cudaStream_t)stream, value);
}

}  // namespace fconv
