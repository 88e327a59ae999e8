// Host side of the C ABI declared in include/gqa_attn.h: argument checks, mode
// resolution, launch planning, the call's own workspace, the K and V tensor
// maps and dispatch to the fused attention and split-combine kernels.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <map>
#include <mutex>
#include <string>

#include "gqa_attn.h"
#include "gqa_attn_kernel.cuh"

namespace gqa_av {
namespace {

constexpr size_t kAttnHeaderBytes = 256;             // device status word + padding
constexpr long long kAttnTimeoutNs = 2000000000LL;   // 2 s bound on every mbarrier wait
constexpr int kAttnMaxSplitRows = 8192;              // longest split of one CTA

thread_local std::string g_at_error;
std::mutex g_at_mu;

int afail(int status, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_at_error = buf;
  return status;
}

int afail_cuda(cudaError_t e, const char* what) {
  return afail(GQA_AV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

using AttnKernel = void (*)(AttnParams);

// The kernel compiled for at most MW consumer warps (6: 255 registers a
// thread; 8: 168).
template <typename Tag>
AttnKernel pick(int D, int ncol, int nw) {
  switch (D) {
    case 64: return gqa_attn_kernel<Tag, 64, 64, 8>;
    case 128:
      return nw > 6 ? gqa_attn_kernel<Tag, 128, 128, 8> : gqa_attn_kernel<Tag, 128, 128, 6>;
    case 256: return ncol == 2 ? gqa_attn_kernel<Tag, 256, 128, 6> : gqa_attn_kernel<Tag, 256, 256, 6>;
    default: return nullptr;
  }
}

struct AttnPlan {
  int mode, heads, hgroups, ncol, kt, nw, stages, rows_per_split, nsplit, tiles;
  int balanced, units, ctas, combine;
  int smem, q_off, qstride, bar_off, stage_bytes, merge_bytes;
  size_t ws_bytes;  // split partials only
};

int check_args(int B, int Cmax, int Hq, int Hkv, int D, int kv_dtype, int mode) {
  if (B <= 0 || Cmax <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0)
    return afail(GQA_AV_ERR_INVALID, "sizes must be positive (B=%d Cmax=%d Hq=%d Hkv=%d D=%d)", B,
                 Cmax, Hq, Hkv, D);
  if (Hq % Hkv) return afail(GQA_AV_ERR_INVALID, "Hq=%d is not a multiple of Hkv=%d", Hq, Hkv);
  if (kv_dtype != GQA_AV_BF16 && kv_dtype != GQA_AV_FP16)
    return afail(GQA_AV_ERR_INVALID, "kv_dtype=%d must be GQA_AV_BF16 or GQA_AV_FP16", kv_dtype);
  if (mode < -1 || mode > 1) return afail(GQA_AV_ERR_INVALID, "mode=%d must be -1, 0 or 1", mode);
  if (D != 64 && D != 128 && D != 256)
    return afail(GQA_AV_ERR_UNSUPPORTED, "D=%d must be 64, 128 or 256", D);
  return GQA_AV_OK;
}

int plan(int dev, int B, int Cmax, int Hq, int Hkv, int D, int kv_dtype, int mode, int want_nw,
         int want_nsplit, int split_mode, int want_ncol, bool ragged, AttnPlan* p) {
  int rc = check_args(B, Cmax, Hq, Hkv, D, kv_dtype, mode);
  if (rc) return rc;
  const int G = Hq / Hkv;
  p->mode = mode == GQA_AV_MODE_AUTO ? (G > 1 ? GQA_AV_MODE_GQA : GQA_AV_MODE_PER_HEAD) : mode;
  // GQA: the group's heads, or the fewest equal chunks of at most 16 of them.
  if (p->mode == GQA_AV_MODE_GQA) {
    int k = (G + kAttnMaxHeads - 1) / kAttnMaxHeads;
    while (G % k) ++k;
    p->heads = G / k;
  } else {
    p->heads = 1;
  }
  p->hgroups = Hq / p->heads;
  // Output column blocks: 2 at D = 256 (see the kernel; measured 2 % faster
  // on the MQA shape, with no register spills), else 1.
  p->ncol = want_ncol > 0 ? want_ncol : (D == 256 ? 2 : 1);
  if (p->ncol != 1 && !(p->ncol == 2 && D == 256))
    return afail(GQA_AV_ERR_UNSUPPORTED, "column_blocks=%d: 1, or 2 at D = 256", p->ncol);
  p->kt = p->hgroups * p->ncol;
  p->tiles = p->kt * B;

  cudaDeviceProp prop;
  cudaError_t e = cudaGetDeviceProperties(&prop, dev);
  if (e != cudaSuccess) return afail_cuda(e, "cudaGetDeviceProperties");
  const int sms = prop.multiProcessorCount;

  // Splits: one CTA per SM over the tiles on few-tile shapes, and no split
  // longer than kAttnMaxSplitRows rows (short waves on many-tile shapes).
  const int max_splits = (Cmax + kAttnRows - 1) / kAttnRows;
  long long want = want_nsplit > 0 ? want_nsplit
                                   : std::max<long long>(p->tiles < sms ? sms / p->tiles : 1,
                                                         (Cmax + kAttnMaxSplitRows - 1) /
                                                             kAttnMaxSplitRows);
  want = std::max<long long>(1, std::min<long long>(want, max_splits));
  const int rps0 = static_cast<int>((Cmax + want - 1) / want);
  p->rows_per_split = (rps0 + kAttnRows - 1) / kAttnRows * kAttnRows;
  p->nsplit = (Cmax + p->rows_per_split - 1) / p->rows_per_split;
  // Balanced splits spread the batch's context rows evenly over the same
  // number of CTAs, whatever the lengths: at most units + tiles CTAs have work.
  p->balanced = split_mode == 2 || (split_mode == 0 && ragged && B > 1);
  if (static_cast<long long>(p->tiles) * (p->nsplit + 1) > 0x7fffffffLL)
    return afail(GQA_AV_ERR_UNSUPPORTED, "grid too large");
  p->units = p->tiles * p->nsplit;
  p->ctas = p->balanced ? p->units + p->tiles : p->units;
  p->combine = p->balanced || p->nsplit > 1;
  const int DV = D / p->ncol;
  p->ws_bytes = p->combine ? static_cast<size_t>(p->ctas) * p->heads *
                                 (static_cast<size_t>(DV) * 4 + 8)
                           : 0;

  // Consumer warps and ring: 32-row stages of K and V (128 * D bytes); the
  // ring holds a whole number of stages per warp, at most 192 KiB. Measured
  // on GB300: 8 warps of 3 stages at D = 64, 6 warps of 2 stages at D = 128
  // (a warp overlaps its next stage's load with the current stage's
  // products; 8 warps of 1 stage measured 2-5 % slower on one-wave and
  // many-wave grids alike), 3 warps of 2 stages at D = 256.
  p->stage_bytes = kAttnRows * (D + DV) * 2;
  p->nw = want_nw > 0 ? want_nw : D == 256 ? 3 : D == 64 ? 8 : 6;
  if (p->nw < 1 || p->nw > attn_max_warps(D))
    return afail(GQA_AV_ERR_UNSUPPORTED, "consumer warps %d outside 1..%d for D=%d", p->nw,
                 attn_max_warps(D), D);
  const int ring_budget = 196608;
  const int per_warp = std::max(1, ring_budget / (p->stage_bytes * p->nw));
  p->stages = per_warp * p->nw;
  p->qstride = D * 2 + 16;
  p->q_off = p->stages * p->stage_bytes;
  p->bar_off = p->q_off + 2 * 16 * p->qstride;
  p->smem = p->bar_off + 2 * p->stages * 8 + 16 + 1024;  // + fail flag, alignment slack
  p->merge_bytes = p->nw * p->heads * ((DV + 4) * 4 + 8);
  if (p->merge_bytes > p->stages * p->stage_bytes)
    return afail(GQA_AV_ERR_UNSUPPORTED, "warp merge (%d B) larger than the ring", p->merge_bytes);
  if (p->smem > static_cast<int>(prop.sharedMemPerBlockOptin))
    return afail(GQA_AV_ERR_UNSUPPORTED, "plan needs %d B of shared memory (limit %d)", p->smem,
                 static_cast<int>(prop.sharedMemPerBlockOptin));
  return GQA_AV_OK;
}

struct Ws {
  void* base = nullptr;
  size_t bytes = 0;
};
std::map<int, Ws> g_at_ws;

int workspace(int dev, size_t need, cudaStream_t stream, Ws* out) {
  std::lock_guard<std::mutex> lk(g_at_mu);
  Ws& w = g_at_ws[dev];
  if (w.base && w.bytes >= need) {
    *out = w;
    return GQA_AV_OK;
  }
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(stream, &cs);
  if (e != cudaSuccess) return afail_cuda(e, "cudaStreamIsCapturing");
  if (cs != cudaStreamCaptureStatusNone)
    return afail(GQA_AV_ERR_NOMEM,
                 "workspace must grow to %zu B but the stream is capturing; make one call with "
                 "the largest shape before capture",
                 need);
  const size_t bytes = std::max(need, w.bytes + w.bytes / 2);
  if (w.base) {
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return afail_cuda(e, "cudaDeviceSynchronize");
    cudaFree(w.base);
    w.base = nullptr;
    w.bytes = 0;
  }
  void* p = nullptr;
  e = cudaMalloc(&p, bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return afail(GQA_AV_ERR_NOMEM, "cudaMalloc(%zu) failed: %s", bytes, cudaGetErrorString(e));
  }
  e = cudaMemset(p, 0, kAttnHeaderBytes);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    cudaFree(p);
    return afail_cuda(e, "zeroing the workspace header");
  }
  w.base = p;
  w.bytes = bytes;
  *out = w;
  return GQA_AV_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 g_at_encode = nullptr;

// A KV cache viewed as 4-D {D, Hkv, Cmax, B} (innermost first); box
// {64, 1, 32, 1} in the 128-byte swizzle: one 128-byte line per row and part.
// Rows past Cmax read as zeros.
int encode_kv_map(CUtensorMap* m, const void* x, int B, int Cmax, int Hkv, int D, const char* what) {
  {
    std::lock_guard<std::mutex> lk(g_at_mu);
    if (!g_at_encode) {
      void* f = nullptr;
      cudaDriverEntryPointQueryResult q;
      cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                                       cudaEnableDefault, &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !f)
        return afail(GQA_AV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
      g_at_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
  }
  const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)Cmax, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)Hkv * D * 2,
                                 (cuuint64_t)Cmax * Hkv * D * 2};
  const cuuint32_t box[4] = {64, 1, (cuuint32_t)kAttnRows, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = g_at_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, const_cast<void*>(x), dims,
                           strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return afail(GQA_AV_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled (%s) failed (%d)", what, (int)r);
  return GQA_AV_OK;
}

cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       void** args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace
}  // namespace gqa_av

using namespace gqa_av;

extern "C" int gqa_attn_plan(int B, int Cmax, int Hq, int Hkv, int D, int kv_dtype, int mode,
                             int consumer_warps, int nsplit, int split_mode, int column_blocks,
                             int ragged, int* info, int n_info) {
  g_at_error.clear();
  int rc = check_args(B, Cmax, Hq, Hkv, D, kv_dtype, mode);
  if (rc) return rc;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return afail_cuda(e, "cudaGetDevice");
  AttnPlan pl;
  if (split_mode < 0 || split_mode > 2)
    return afail(GQA_AV_ERR_INVALID, "split_mode=%d must be 0, 1 or 2", split_mode);
  if (column_blocks < 0) return afail(GQA_AV_ERR_INVALID, "column_blocks=%d < 0", column_blocks);
  rc = plan(dev, B, Cmax, Hq, Hkv, D, kv_dtype, mode, consumer_warps, nsplit, split_mode,
            column_blocks, ragged != 0, &pl);
  if (rc) return rc;
  const int vals[] = {pl.mode, pl.heads, pl.nw, pl.stages, pl.rows_per_split, pl.nsplit,
                      pl.tiles, pl.smem, pl.balanced ? 2 : 1, pl.ctas, pl.ncol};
  if (info)
    for (int i = 0; i < n_info && i < static_cast<int>(sizeof vals / sizeof vals[0]); ++i)
      info[i] = vals[i];
  return GQA_AV_OK;
}

extern "C" int gqa_attn_decode_tuned(const float* q, const void* k_cache, const void* v_cache,
                                     const int32_t* seq_lens, float* out, int B, int Cmax, int Hq,
                                     int Hkv, int D, int kv_dtype, float scale, int mode,
                                     int consumer_warps, int nsplit, int split_mode,
                                     int column_blocks, void* stream_) {
  g_at_error.clear();
  if (!q || !k_cache || !v_cache || !out)
    return afail(GQA_AV_ERR_INVALID, "q, k_cache, v_cache and out must be non-NULL");
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_cache) |
       reinterpret_cast<uintptr_t>(v_cache) | reinterpret_cast<uintptr_t>(out)) & 15u)
    return afail(GQA_AV_ERR_UNSUPPORTED, "q, k_cache, v_cache and out must be 16-byte aligned");
  if (!std::isfinite(scale)) return afail(GQA_AV_ERR_INVALID, "scale must be finite");
  int rc = check_args(B, Cmax, Hq, Hkv, D, kv_dtype, mode);
  if (rc) return rc;
  if (consumer_warps < 0 || consumer_warps > kAttnMaxWarps || nsplit < 0 || split_mode < 0 ||
      split_mode > 2 || column_blocks < 0)
    return afail(GQA_AV_ERR_INVALID,
                 "consumer_warps=%d (0..%d), nsplit=%d (>= 0), split_mode=%d (0..2) or "
                 "column_blocks=%d (>= 0) out of range",
                 consumer_warps, kAttnMaxWarps, nsplit, split_mode, column_blocks);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return afail_cuda(e, "cudaGetDevice");
  AttnPlan pl;
  if ((rc = plan(dev, B, Cmax, Hq, Hkv, D, kv_dtype, mode, consumer_warps, nsplit, split_mode,
                 column_blocks, seq_lens != nullptr, &pl)))
    return rc;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  Ws ws;
  if ((rc = workspace(dev, kAttnHeaderBytes + pl.ws_bytes, stream, &ws))) return rc;

  AttnParams p;
  if ((rc = encode_kv_map(&p.k_map, k_cache, B, Cmax, Hkv, D, "K"))) return rc;
  if ((rc = encode_kv_map(&p.v_map, v_cache, B, Cmax, Hkv, D, "V"))) return rc;
  p.q = q;
  p.seq_lens = seq_lens;
  p.out = out;
  p.status = static_cast<unsigned int*>(ws.base);
  char* parts = static_cast<char*>(ws.base) + kAttnHeaderBytes;
  p.ws_o = reinterpret_cast<float*>(parts);
  p.ws_ml = reinterpret_cast<float2*>(parts + static_cast<size_t>(pl.ctas) * pl.heads *
                                                  (D / pl.ncol) * 4);
  p.qscale = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);  // log2(e)
  p.B = B; p.Cmax = Cmax; p.Hq = Hq; p.Hkv = Hkv; p.D = D; p.G = Hq / Hkv;
  p.heads = pl.heads; p.hgroups = pl.hgroups; p.nw = pl.nw; p.stages = pl.stages;
  p.ncol = pl.ncol; p.kt = pl.kt;
  p.rows_per_split = pl.rows_per_split; p.nsplit = pl.nsplit;
  p.balanced = pl.balanced; p.units = pl.units;
  p.stage_bytes = static_cast<uint32_t>(pl.stage_bytes);
  p.q_off = static_cast<uint32_t>(pl.q_off);
  p.qstride = static_cast<uint32_t>(pl.qstride);
  p.bar_off = static_cast<uint32_t>(pl.bar_off);
  p.timeout_ns = kAttnTimeoutNs;

  AttnKernel k = kv_dtype == GQA_AV_BF16 ? pick<Bf16Tag>(D, pl.ncol, pl.nw)
                                         : pick<Fp16Tag>(D, pl.ncol, pl.nw);
  if (!k) return afail(GQA_AV_ERR_UNSUPPORTED, "no attention kernel for D=%d", D);
  e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, pl.smem);
  if (e != cudaSuccess) return afail_cuda(e, "cudaFuncSetAttribute");
  void* args1[] = {&p};
  e = launch_pdl(reinterpret_cast<const void*>(k), dim3(pl.ctas),
                 dim3(32 * (pl.nw + 1)), pl.smem, stream, args1);
  if (e != cudaSuccess) return afail_cuda(e, "attention kernel launch");
  if (!pl.combine) return GQA_AV_OK;  // every tile wrote `out` itself

  AttnCombineParams c;
  c.ws_o = p.ws_o;
  c.ws_ml = p.ws_ml;
  c.seq_lens = seq_lens;
  c.out = out;
  c.B = B; c.Cmax = Cmax; c.Hq = Hq; c.D = D; c.heads = pl.heads; c.hgroups = pl.hgroups;
  c.rows_per_split = pl.rows_per_split; c.nsplit = pl.nsplit;
  c.balanced = pl.balanced; c.units = pl.units;
  c.ncol = pl.ncol; c.kt = pl.kt;
  void* args2[] = {&c};
  e = launch_pdl(reinterpret_cast<const void*>(gqa_attn_combine_kernel), dim3(pl.tiles * pl.heads),
                 dim3(kAttnCombineThreads), 0, stream, args2);
  if (e != cudaSuccess) return afail_cuda(e, "combine kernel launch");
  return GQA_AV_OK;
}

extern "C" int gqa_attn_decode(const float* q, const void* k_cache, const void* v_cache,
                               const int32_t* seq_lens, float* out, int B, int Cmax, int Hq,
                               int Hkv, int D, int kv_dtype, float scale, int mode, void* stream) {
  return gqa_attn_decode_tuned(q, k_cache, v_cache, seq_lens, out, B, Cmax, Hq, Hkv, D, kv_dtype,
                               scale, mode, 0, 0, 0, 0, stream);
}

extern "C" int gqa_attn_device_status(void* stream_, int clear) {
  g_at_error.clear();
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return afail_cuda(e, "cudaGetDevice");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return afail_cuda(e, "cudaStreamSynchronize");
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_at_mu);
    auto it = g_at_ws.find(dev);
    if (it != g_at_ws.end()) base = it->second.base;
  }
  if (!base) return GQA_AV_OK;
  unsigned word = 0;
  e = cudaMemcpy(&word, base, sizeof word, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return afail_cuda(e, "reading the status word");
  if (word && clear) {
    e = cudaMemset(base, 0, sizeof word);
    if (e != cudaSuccess) return afail_cuda(e, "clearing the status word");
  }
  if (word)
    return afail(GQA_AV_ERR_DEVICE_TIMEOUT, "a bounded wait in the attention kernel ran out (0x%x)",
                 word);
  return GQA_AV_OK;
}

extern "C" const char* gqa_attn_last_error(void) { return g_at_error.c_str(); }
