// Internal interface between the planner (fconv_api.cpp) and the CUDA launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <utility>

#include "../../include/fconv.h"

namespace fconv {

// Resolved geometry of one FusedConv call. Spatial axes are (depth, height, width);
// axes the rank lacks have extent 1, stride 1, dilation 1 and pad 0. Pads are the
// begin pads actually applied (manifest derive effectivePadFront/Top/Left).
struct ConvGeom {
  int dtype;                    // fconv_dtype
  int N, C, M, G, Cg, Mg;
  int ID, IH, IW;
  int OD, OH, OW;
  int KD, KH, KW;
  int sD, sH, sW;
  int dD, dH, dW;
  int pD, pH, pW;
  int act;                      // fconv_act
  float alpha, beta;            // resolved activation parameters
  int has_bias, has_z;
  long long P;                  // OD*OH*OW
  long long IS;                 // ID*IH*IW
  int KV;                       // KD*KH*KW
  int Kg;                       // Cg*KV
  int max_ctas;                 // cap on persistent CTAs (0 = none)
  int transposed;               // transposed convolution (W is (C, M/group, kernel...))
  int precision;                // fconv_precision
};

struct ConvArgs {
  const void* x;
  const void* w;
  const void* b;
  const void* z;
  void* y;
  void* ws;
};

// Tensor-core implicit GEMM configuration.
struct IgemmConfig {
  int tile_n;      // largest pixel tile (MMA N): 64, 128 or 256; channel tiles are 128
  int split_k;     // number of K splits (>= 1)
  long long grid;  // persistent CTAs (one per SM at most)
  int a_path;      // 1: im2col rows built in-kernel from the NC(D)HW input patch
                   //    (k_igemm_patch.cu); 2: TMA boxes of X repacked in 64-channel blocks
                   //    (k_igemm_tc.cu)
};

// Launchers: return cudaError_t as int (0 = success).
int launch_direct(const ConvGeom& g, const ConvArgs& a, void* stream);
int launch_depthwise(const ConvGeom& g, const ConvArgs& a, void* stream);
bool depthwise_supported(const ConvGeom& g);
bool depthwise_half2_supported(const ConvGeom& g);
int read_and_clear_dw_error(void* stream, unsigned* value);
int launch_grouped(const ConvGeom& g, const ConvArgs& a, void* stream);
bool grouped_supported(const ConvGeom& g);
int read_and_clear_grouped_error(void* stream, unsigned* value);
int launch_transposed(const ConvGeom& g, const ConvArgs& a, void* stream);
bool transposed_supported(const ConvGeom& g);

// tcgen05 implicit GEMM: dispatch between the two A paths (k_igemm_tc.cu).
int launch_igemm_tc(const ConvGeom& g, const IgemmConfig& c, const ConvArgs& a, void* stream);
bool igemm_tc_supported(const ConvGeom& g, int max_px);    // some im2col path runs the request
bool igemm_tc_tma_capable(const ConvGeom& g);             // the TMA-fed path runs it
// The im2col path for a request (0 auto, 1 patch, 2 TMA-fed): 1 or 2, or 0 when none can.
int igemm_tc_resolve_path(const ConvGeom& g, int max_px, int requested);
size_t igemm_tc_workspace_bytes(const ConvGeom& g, const IgemmConfig& c);
long long igemm_tc_mtiles(const ConvGeom& g, int a_path, int max_px);  // pixel tiles
int igemm_tc_chunks(const ConvGeom& g, int a_path, int max_px);        // 64-wide K chunks
int igemm_tc_launches(const ConvGeom& g, const IgemmConfig& c);  // kernels per fconv_run
int launch_splitk_reduce(const ConvGeom& g, int splits, const float* part, const void* b,
                         const void* z, void* y, void* stream);

// The patch-fed kernel (k_igemm_patch.cu).
bool igemm_patch_capable(const ConvGeom& g, int tile_n);
long long igemm_patch_mtiles(const ConvGeom& g, int tile_n);
int igemm_patch_chunks(const ConvGeom& g, int tile_n);
size_t igemm_patch_workspace_bytes(const ConvGeom& g, const IgemmConfig& c);
int igemm_patch_launches(const ConvGeom& g, const IgemmConfig& c);
int launch_igemm_patch(const ConvGeom& g, const IgemmConfig& c, const ConvArgs& a, void* stream);
int read_and_clear_patch_error(void* stream, unsigned* value);

// The fp32 3xTF32 kernel (k_igemm_tf32.cu): C/group a multiple of 32.
bool igemm_tf32_capable(const ConvGeom& g, int max_px);
long long igemm_tf32_mtiles(const ConvGeom& g, int max_px);
int igemm_tf32_chunks(const ConvGeom& g);
size_t igemm_tf32_workspace_bytes(const ConvGeom& g, const IgemmConfig& c);
int launch_igemm_tf32(const ConvGeom& g, const IgemmConfig& c, const ConvArgs& a, void* stream);
int read_and_clear_tf32_error(void* stream, unsigned* value);

// cuTensorMapEncodeTiled from the driver (null when unavailable).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn tensor_map_encoder();

// Launch with programmatic stream serialization: the kernel may begin (and run up to its
// pdl_wait()) while the previous kernel in the stream finishes.
template <typename... KArgs, typename... Args>
inline int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                      void* stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = (cudaStream_t)stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return (int)cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Device error word (set by kernels whose bounded waits gave up). Reads and clears.
int read_and_clear_device_error(void* stream, unsigned* value);

}  // namespace fconv
