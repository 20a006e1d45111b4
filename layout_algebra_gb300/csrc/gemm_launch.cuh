// Host launchers of the GEMM kernel instances (included by gemm_inst.cu only).
#pragma once

#include "gemm_kernel.cuh"

namespace gb {

template <bool kBF16, int kIn, int kShape>
gb_status prepare_single(DeviceState* dev) {
  using C = gb::Cfg<false, kIn, kShape>;
  bool& smem_set = dev->attr_single[kBF16][kIn][kShape == gb::kShapeNarrow];
  if (!smem_set) {
    if (cudaFuncSetAttribute(gb::gemm_kernel<kBF16, false, kIn, kShape>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes) != cudaSuccess)
      return GB_ERR_LAUNCH;
    smem_set = true;
  }
  return GB_OK;
}

template <bool kBF16, int kIn, int kShape>
gb_status launch_single(const Maps& m, const Params& p, int grid, cudaStream_t s) {
  using C = gb::Cfg<false, kIn, kShape>;
  // programmatic stream serialisation: the kernel's set-up may overlap the end of the previous
  // kernel in the stream (it waits for that kernel before touching global memory)
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(C::kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, gb::gemm_kernel<kBF16, false, kIn, kShape>, m.a, m.b, m.sfa, m.sfb, m.c, m.d, m.at,
                         m.bt, p) != cudaSuccess)
    return GB_ERR_LAUNCH;
  return cudaGetLastError() == cudaSuccess ? GB_OK : GB_ERR_LAUNCH;
}

template <bool kBF16, int kIn, int kShape>
gb_status prepare_pair(DeviceState* dev) {
  using C = gb::Cfg<true, kIn, kShape>;
  constexpr int kCl = 2;   // CTAs per cluster: one pair
  bool& attr = dev->attr_pair[kBF16][kIn][pair_shape_index(kShape)];
  if (!attr) {
    if (cudaFuncSetAttribute(gb::gemm_kernel<kBF16, true, kIn, kShape>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes) != cudaSuccess)
      return GB_ERR_LAUNCH;
    attr = true;
  }
  int& clusters = dev->pair_clusters[pair_shape_index(kShape)];
  if (clusters == 0) {
    // a persistent grid must fit at once: ask how many clusters can be resident together
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = kCl;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(C::kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(kCl * (dev->sms / kCl), 1, 1);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gb::gemm_kernel<kBF16, true, kIn, kShape>, &cfg) != cudaSuccess ||
        n <= 0)
      n = dev->sms / kCl;
    clusters = std::min(n, dev->sms / kCl);
  }
  return GB_OK;
}

template <bool kBF16, int kIn, int kShape>
gb_status launch_pair(const Maps& m, const Params& p, int clusters, cudaStream_t s) {
  using C = gb::Cfg<true, kIn, kShape>;
  constexpr int kCl = 2;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // programmatic stream serialisation (see launch_single)
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(C::kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cfg.gridDim = dim3(kCl * clusters, 1, 1);
  if (cudaLaunchKernelEx(&cfg, gb::gemm_kernel<kBF16, true, kIn, kShape>, m.a, m.b, m.sfa, m.sfb, m.c, m.d, m.at, m.bt, p) != cudaSuccess)
    return GB_ERR_LAUNCH;
  return cudaGetLastError() == cudaSuccess ? GB_OK : GB_ERR_LAUNCH;
}

}  // namespace gb
