// Explicit instantiations of the AV kernel for one V element type.
// Included by gqa_av_bf16.cu / gqa_av_fp16.cu with GQA_AV_TAG defined, so the
// two element types compile as separate translation units in parallel.
#pragma once
#include "gqa_av_kernel.cuh"
#include "gqa_av_mma.cuh"
#include "gqa_av_stream.cuh"

namespace gqa_av {

// Launched with programmatic stream serialization: the kernel's prologue may
// overlap the previous kernel's tail; it waits (griddepcontrol.wait) before it
// touches data of earlier kernels.
template <typename Tag, int GC>
cudaError_t launch(const Params& p, int grid, int smem_bytes, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(cta_threads(GC));
  cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, gqa_av_kernel<Tag, GC>, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// Raises the kernel's dynamic shared-memory limit to `smem_limit` (the device's
// opt-in maximum, so every plan can launch) and reports CTAs per SM at `smem_bytes`.
template <typename Tag, int GC>
cudaError_t occupancy(int smem_limit, int smem_bytes, int* ctas_per_sm) {
  cudaError_t e = cudaFuncSetAttribute(gqa_av_kernel<Tag, GC>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem_limit);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, gqa_av_kernel<Tag, GC>,
                                                       cta_threads(GC), smem_bytes);
}

// The same for the tensor-core kernel, NB = N / 16 blocks of 16 heads.
template <typename Tag, int NB>
cudaError_t launch_mma(const Params& p, int grid, int smem_bytes, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(mma_threads(p.cvt_warps));
  cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, gqa_av_mma_kernel<Tag, NB>, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <typename Tag, int NB>
cudaError_t occupancy_mma(int smem_limit, int smem_bytes, int* ctas_per_sm) {
  cudaError_t e = cudaFuncSetAttribute(gqa_av_mma_kernel<Tag, NB>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem_limit);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, gqa_av_mma_kernel<Tag, NB>,
                                                       kMmaMaxThreads, smem_bytes);
}

// The streamed tensor-core kernel: one persistent CTA per SM (or more).
template <typename Tag, int NB>
cudaError_t launch_stream(const Params& p, int grid, int smem_bytes, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(mma_threads(p.cvt_warps));
  cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, gqa_av_stream_kernel<Tag, NB>, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <typename Tag, int NB>
cudaError_t occupancy_stream(int smem_limit, int smem_bytes, int* ctas_per_sm) {
  cudaError_t e = cudaFuncSetAttribute(gqa_av_stream_kernel<Tag, NB>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem_limit);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, gqa_av_stream_kernel<Tag, NB>,
                                                       kMmaMaxThreads, smem_bytes);
}

#define GQA_AV_INSTANTIATE_STREAM(TAG, NB)                                               \
  template cudaError_t launch_stream<TAG, NB>(const Params&, int, int, cudaStream_t);    \
  template cudaError_t occupancy_stream<TAG, NB>(int, int, int*);

#define GQA_AV_INSTANTIATE_MMA(TAG, NB)                                                  \
  template cudaError_t launch_mma<TAG, NB>(const Params&, int, int, cudaStream_t);       \
  template cudaError_t occupancy_mma<TAG, NB>(int, int, int*);

#define GQA_AV_INSTANTIATE(TAG, GC)                                                      \
  template cudaError_t launch<TAG, GC>(const Params&, int, int, cudaStream_t);           \
  template cudaError_t occupancy<TAG, GC>(int, int, int*);

#define GQA_AV_INSTANTIATE_ALL(TAG) \
  GQA_AV_INSTANTIATE(TAG, 1)        \
  GQA_AV_INSTANTIATE(TAG, 2)        \
  GQA_AV_INSTANTIATE(TAG, 3)        \
  GQA_AV_INSTANTIATE(TAG, 4)        \
  GQA_AV_INSTANTIATE(TAG, 5)        \
  GQA_AV_INSTANTIATE(TAG, 6)        \
  GQA_AV_INSTANTIATE(TAG, 7)        \
  GQA_AV_INSTANTIATE(TAG, 8)        \
  GQA_AV_INSTANTIATE(TAG, 12)       \
  GQA_AV_INSTANTIATE_MMA(TAG, 1)    \
  GQA_AV_INSTANTIATE_MMA(TAG, 2)    \
  GQA_AV_INSTANTIATE_MMA(TAG, 3)    \
  GQA_AV_INSTANTIATE_MMA(TAG, 4)    \
  GQA_AV_INSTANTIATE_STREAM(TAG, 1) \
  GQA_AV_INSTANTIATE_STREAM(TAG, 2) \
  GQA_AV_INSTANTIATE_STREAM(TAG, 3) \
  GQA_AV_INSTANTIATE_STREAM(TAG, 4)

}  // namespace gqa_av
