// gqa_av_decode_noalloc: the AV reduction for callers that cannot allocate
// device memory.
//
// Some callers may not call cudaMalloc/cudaFree at the moment they run the
// reduction. Examples:
//   * plug-ins inside an inference engine that owns every byte of device
//     memory and forbids allocation while it enqueues work;
//   * latency-critical decode loops that must never hit the implicit device
//     synchronisation a cudaFree (or a growing allocation) can cause;
//   * processes that reserve their whole memory budget up front.
// gqa_av_decode keeps a growable workspace and may allocate on a call that
// needs more of it. This entry point instead keeps its scratch (status word,
// split partials) in the fixed file-scope array below, so no call ever
// allocates.
//
// The array holds GQA_AV_NOALLOC_SCRATCH_BYTES on every GPU that loads this
// library, until the process exits. Its device address is looked up once per
// device, by that device's first call, with cudaGetSymbolAddress; the same
// set-up zeroes the status word and registers its address, so that
// gqa_av_device_status reports (and clears) a bounded wait that ran out in
// one of these calls. Host code must not use the array's name as a device
// address: on the host that name is a stand-in. All calls on a device share
// the array and it keeps the last call's contents: the status word is never
// cleared by a call (a later call would otherwise hide an earlier timeout),
// and split partials are always written before they are read. Calls that may
// overlap on the GPU (different streams, no ordering between them) race on it.
#include <cuda_runtime.h>

#include <map>
#include <mutex>

#include "gqa_av.h"

namespace gqa_av {
int record_error(int status, const char* msg);
void register_noalloc_status(int dev, void* status_word);
int run_in_scratch(const float* attn, const void* v, const int32_t* seq_lens, float* out, int B,
                   int Cmax, int Hq, int Hkv, int D, int v_dtype, int mode, cudaStream_t stream,
                   void* scratch, size_t status_bytes, size_t scratch_bytes);
}  // namespace gqa_av

namespace {

constexpr size_t kScratchBytes = GQA_AV_NOALLOC_SCRATCH_BYTES;
constexpr size_t kStatusBytes = 256;  // device status word + padding; partials follow
static_assert(kStatusBytes < kScratchBytes, "scratch too small");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
std::map<int, void*> g_scratch_addr;  // device -> device address of g_noalloc_scratch

// Set-up, once per device, with that device current.
int scratch_address(int dev, void** out) {
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_scratch_addr.find(dev);
  if (it != g_scratch_addr.end()) {
    *out = it->second;
    return GQA_AV_OK;
  }
  void* ptr = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
  if (e != cudaSuccess || ptr == nullptr)
    return gqa_av::record_error(GQA_AV_ERR_CUDA,
                                "cudaGetSymbolAddress of the no-allocation scratch failed");
  // The status word starts at zero; from here on only gqa_av_device_status clears it.
  e = cudaMemset(ptr, 0, kStatusBytes);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess)
    return gqa_av::record_error(GQA_AV_ERR_CUDA,
                                "zeroing the no-allocation status word failed");
  gqa_av::register_noalloc_status(dev, ptr);
  g_scratch_addr[dev] = ptr;
  *out = ptr;
  return GQA_AV_OK;
}

}  // namespace

namespace gqa_av {
// The fixed array of this device (set up on first use): its address, the
// bytes of its status-word header, and its size.
int noalloc_scratch(int dev, void** ptr, size_t* status_bytes, size_t* bytes) {
  int rc = scratch_address(dev, ptr);
  if (rc) return rc;
  *status_bytes = kStatusBytes;
  *bytes = kScratchBytes;
  return GQA_AV_OK;
}
}  // namespace gqa_av

extern "C" int gqa_av_decode_noalloc(const float* attn, const void* v_cache,
                                     const int32_t* seq_lens, float* out, int B, int Cmax, int Hq,
                                     int Hkv, int D, int v_dtype, int mode, void* stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return gqa_av::record_error(GQA_AV_ERR_CUDA, "cudaGetDevice failed");
  void* scratch = nullptr;
  int rc = scratch_address(dev, &scratch);
  if (rc) return rc;
  return gqa_av::run_in_scratch(attn, v_cache, seq_lens, out, B, Cmax, Hq, Hkv, D, v_dtype, mode,
                                static_cast<cudaStream_t>(stream), scratch, kStatusBytes,
                                kScratchBytes);
}
