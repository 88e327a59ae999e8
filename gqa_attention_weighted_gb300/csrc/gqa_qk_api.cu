// Host side of the C ABI declared in include/gqa_qk.h: argument checks, mode
// resolution, launch planning, the call's own workspace, the K tensor map and
// dispatch to the score and normalise kernels.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <map>
#include <mutex>
#include <string>

#include "gqa_qk.h"
#include "gqa_qk_kernel.cuh"
#include "gqa_qk_mma.cuh"
#include "gqa_qk_stream.cuh"

namespace gqa_av {
namespace {

constexpr size_t kQkHeaderBytes = 256;              // device status word + padding
constexpr long long kQkTimeoutNs = 2000000000LL;    // 2 s bound on every mbarrier wait

thread_local std::string g_qk_error;
std::mutex g_qk_mu;

int qfail(int status, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_qk_error = buf;
  return status;
}

int qfail_cuda(cudaError_t e, const char* what) {
  return qfail(GQA_AV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

using QkKernel = void (*)(QkParams);

template <typename Tag>
QkKernel pick(int gc) {
  switch (gc) {
    case 1: return gqa_qk_kernel<Tag, 1>;
    case 2: return gqa_qk_kernel<Tag, 2>;
    case 3: return gqa_qk_kernel<Tag, 3>;
    case 4: return gqa_qk_kernel<Tag, 4>;
    case 5: return gqa_qk_kernel<Tag, 5>;
    case 6: return gqa_qk_kernel<Tag, 6>;
    case 7: return gqa_qk_kernel<Tag, 7>;
    case 8: return gqa_qk_kernel<Tag, 8>;
    case 9: return gqa_qk_kernel<Tag, 9>;
    case 10: return gqa_qk_kernel<Tag, 10>;
    case 11: return gqa_qk_kernel<Tag, 11>;
    case 12: return gqa_qk_kernel<Tag, 12>;
    case 13: return gqa_qk_kernel<Tag, 13>;
    case 14: return gqa_qk_kernel<Tag, 14>;
    case 15: return gqa_qk_kernel<Tag, 15>;
    case 16: return gqa_qk_kernel<Tag, 16>;
    default: return nullptr;
  }
}

template <typename Tag>
QkKernel pick_stream(int nb) {
  switch (nb) {
    case 1: return gqa_qk_stream_kernel<Tag, 1>;
    case 2: return gqa_qk_stream_kernel<Tag, 2>;
    case 3: return gqa_qk_stream_kernel<Tag, 3>;
    case 4: return gqa_qk_stream_kernel<Tag, 4>;
    default: return nullptr;
  }
}

template <typename Tag>
QkKernel pick_mma(int nb) {
  switch (nb) {
    case 1: return gqa_qk_mma_kernel<Tag, 1>;
    case 2: return gqa_qk_mma_kernel<Tag, 2>;
    case 3: return gqa_qk_mma_kernel<Tag, 3>;
    case 4: return gqa_qk_mma_kernel<Tag, 4>;
    default: return nullptr;
  }
}

// Engines: the CUDA-core FMA kernel, the tcgen05 kernel with fixed splits,
// and the streamed tcgen05 kernel (the default where it applies).
constexpr int kQkEngineFma = 1, kQkEngineTensor = 2, kQkEngineStream = 3;
constexpr int kQkStreamStages = 2;  // K ring depth of the streamed score kernel

struct QkPlan {
  int engine, npad, b_off, tmem_cols, threads;
  int split_units, lens_off;  // streamed kernel
  size_t whole_off;           // streamed kernel: byte offset of the whole-tile pairs
  int mode, heads, hgroups, gc, nc, rs, R, stages, parts, rows_per_split, nsplit, tiles;
  int smem, q_off, red_off, bar_off, stage_bytes;
  int norm_rows, norm_ctas_per_b;
  size_t ws_bytes;  // per-split pairs only
};

// Argument checks that need no CUDA call.
int check_args(int B, int Cmax, int Hq, int Hkv, int D, int k_dtype, int mode) {
  if (B <= 0 || Cmax <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0)
    return qfail(GQA_AV_ERR_INVALID, "sizes must be positive (B=%d Cmax=%d Hq=%d Hkv=%d D=%d)", B,
                 Cmax, Hq, Hkv, D);
  if (Hq % Hkv) return qfail(GQA_AV_ERR_INVALID, "Hq=%d is not a multiple of Hkv=%d", Hq, Hkv);
  if (k_dtype != GQA_AV_BF16 && k_dtype != GQA_AV_FP16)
    return qfail(GQA_AV_ERR_INVALID, "k_dtype=%d must be GQA_AV_BF16 or GQA_AV_FP16", k_dtype);
  if (mode < -1 || mode > 1) return qfail(GQA_AV_ERR_INVALID, "mode=%d must be -1, 0 or 1", mode);
  if (D != 64 && D != 128 && D != 256)
    return qfail(GQA_AV_ERR_UNSUPPORTED, "D=%d must be 64, 128 or 256", D);
  if (Hq > kQkMaxHeads * 32) return qfail(GQA_AV_ERR_UNSUPPORTED, "Hq=%d above 2048", Hq);
  return GQA_AV_OK;
}

// CTAs of `threads` threads and `smem` bytes of dynamic shared memory that
// one SM holds by its shared memory, registers and threads (registers are
// given out per warp in units of 256).
int resident_ctas(const void* fn, int threads, int smem, const cudaDeviceProp& prop) {
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess) return 0;
  const int warps = (threads + 31) / 32;
  const long long regs_cta = (static_cast<long long>(fa.numRegs) * 32 + 255) / 256 * 256 * warps;
  const long long smem_cta =
      static_cast<long long>(smem) + fa.sharedSizeBytes + prop.reservedSharedMemPerBlock;
  long long n = prop.maxThreadsPerMultiProcessor / (32LL * warps);
  if (regs_cta > 0) n = std::min(n, prop.regsPerMultiprocessor / regs_cta);
  if (smem_cta > 0) n = std::min<long long>(n, static_cast<long long>(prop.sharedMemPerMultiprocessor) / smem_cta);
  return static_cast<int>(n);
}

// Normalise launch: a CTA rewrites `norm_rows` rows of one sequence, in
// batches of qk_norm_rows_per_batch(Hq) rows (the next batch's loads in
// flight while the current one is written). One batch a CTA where that
// makes one wave (kQkNormCtasPerSm an SM) or less: the latency-bound short
// calls; on longer calls as many batches a CTA (up to kQkNormMaxIters) as
// keep the grid near one wave, so the pair loads and merges of a CTA are paid
// once for many rows. Measured on GB300 (us per call of the score step, grid
// of about 10 / 4 / 2 / 1 CTAs an SM): MQA-style 30.7 / 29.8 / 31.9 / 35.8,
// the 32-sequence ragged batch 142.9 / 140.6 / 156.6 / 188.9; with one batch
// a CTA the ragged batch's 79 MB of scores took 93 us to rewrite. At most 8
// batches a CTA (against 64 / 32 / 16): the large ragged batch 1276 us (1334
// / 1296 / 1281), whose long blocks past a sequence's length left CTAs idle.
void norm_layout(QkPlan* p, int B, int Cmax, int Hq, int sms) {
  const int base = qk_norm_rows_per_batch(Hq);
  const long long blocks = static_cast<long long>(B) * ((Cmax + base - 1) / base);
  const long long target = 1LL * kQkNormCtasPerSm * sms;
  const long long iters = std::min<long long>(kQkNormMaxIters, std::max<long long>(1, (blocks + target - 1) / target));
  p->norm_rows = base * static_cast<int>(iters);
  p->norm_ctas_per_b = (Cmax + p->norm_rows - 1) / p->norm_rows;
}

int plan(int dev, int B, int Cmax, int Hq, int Hkv, int D, int k_dtype, int mode, int engine,
         QkPlan* p) {
  int rc = check_args(B, Cmax, Hq, Hkv, D, k_dtype, mode);
  if (rc) return rc;
  if (engine < 0 || engine > kQkEngineStream)
    return qfail(GQA_AV_ERR_INVALID,
                 "engine=%d must be 0 (auto), 1 (FMA), 2 (tensor, fixed splits) or 3 (streamed)",
                 engine);
  // The streamed tensor-core kernel is the default except on short streams
  // with fewer tiles (sequences x head groups) than SMs, where the
  // fixed-split kernel runs about two CTAs an SM in one wave (D <= 128 and at
  // most 2048 x 2 x SMs tile rows). Measured on GB300, us per call, fixed vs
  // streamed: Llama-size 12.8 vs 14.7 and Phi-style 26.1 vs 27.3 (short);
  // MQA-style 40.6 vs 39.9 (D = 256), the 4x-L2 traffic shape 123 vs 98, its
  // 32-sequence ragged twin 235 vs 157. The streamed kernel keeps the lengths
  // in shared memory (at most kStreamMaxB sequences).
  if (engine == kQkEngineStream && B > kStreamMaxB)
    return qfail(GQA_AV_ERR_UNSUPPORTED, "the streamed kernel takes at most %d sequences",
                 kStreamMaxB);
  {
    const int G0 = Hq / Hkv;
    const int heads0 = (mode == GQA_AV_MODE_GQA || (mode == GQA_AV_MODE_AUTO && G0 > 1)) ? G0 : 1;
    int sms0 = 0;
    cudaError_t e0 = cudaDeviceGetAttribute(&sms0, cudaDevAttrMultiProcessorCount, dev);
    if (e0 != cudaSuccess) return qfail_cuda(e0, "cudaDeviceGetAttribute");
    const long long tiles0 = static_cast<long long>(B) * (Hq / heads0);
    const bool short_few = tiles0 < sms0 && D <= 128 && tiles0 * Cmax <= 2048LL * 2 * sms0;
    p->engine = engine ? engine
                       : (B <= kStreamMaxB && !short_few ? kQkEngineStream : kQkEngineTensor);
  }
  const bool auto_stream = engine == 0 && p->engine == kQkEngineStream;
  const int G = Hq / Hkv;
  p->mode = mode == GQA_AV_MODE_AUTO ? (G > 1 ? GQA_AV_MODE_GQA : GQA_AV_MODE_PER_HEAD) : mode;
  p->heads = p->mode == GQA_AV_MODE_GQA ? G : 1;
  if (p->heads > kQkMaxHeads)
    return qfail(GQA_AV_ERR_UNSUPPORTED, "%d heads per KV head, at most %d", p->heads, kQkMaxHeads);
  p->hgroups = Hq / p->heads;
  // Head chunks: the fewest of 1, 2, 4, 8 that leave at most 16 heads a thread.
  p->nc = 0;
  for (int nc = 1; nc <= 8; nc *= 2)
    if (p->heads % nc == 0 && p->heads / nc <= 16) { p->nc = nc; break; }
  if (!p->nc)
    return qfail(GQA_AV_ERR_UNSUPPORTED, "%d heads per CTA do not split into <= 8 chunks of <= 16",
                 p->heads);
  p->gc = p->heads / p->nc;
  p->rs = kQkConsumerThreads / p->nc;
  p->parts = D / 64;
  const bool tensor = p->engine == kQkEngineTensor || p->engine == kQkEngineStream;
  if (tensor) {
    // 128 context rows (the MMA's M) a stage; N = 2 x heads padded to 16.
    p->R = kQkMmaRows;
    p->npad = (p->heads + 15) / 16 * 16;
    p->tmem_cols = 32;
    while (p->tmem_cols < 4 * p->npad) p->tmem_cols *= 2;
    p->threads = p->engine == kQkEngineStream ? kQkStreamThreads : kQkMmaThreads;
  } else {
    // One K row per consumer thread and stage, at most 64 KiB a stage, a
    // multiple of 32 rows so a warp is busy or idle as a whole.
    p->R = std::min(p->rs, 32768 / D) / 32 * 32;
    p->npad = 0;
    p->tmem_cols = 0;
    p->threads = kQkThreads;
  }
  p->stage_bytes = p->R * D * 2;

  cudaDeviceProp prop;
  cudaError_t e = cudaGetDeviceProperties(&prop, dev);
  if (e != cudaSuccess) return qfail_cuda(e, "cudaGetDeviceProperties");
  const int sms = prop.multiProcessorCount;
  const int optin = static_cast<int>(prop.sharedMemPerBlockOptin);

  p->tiles = p->hgroups * B;
  if (p->engine == kQkEngineStream) {
    // Two CTAs an SM where two fit (registers and shared memory; one at
    // D = 256, whose 64 KiB stages need the room), in groups of one CTA per
    // head group, each with a ring of two 128-row stages.
    QkKernel kfn = k_dtype == GQA_AV_BF16 ? pick_stream<Bf16Tag>(p->npad / 16)
                                          : pick_stream<Fp16Tag>(p->npad / 16);
    if (!kfn) return qfail(GQA_AV_ERR_UNSUPPORTED, "no score kernel for this head count");
    // All of the SM's unified memory as shared memory, so two CTAs fit.
    cudaError_t e2 = cudaFuncSetAttribute(kfn, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e2 != cudaSuccess) return qfail_cuda(e2, "cudaFuncSetAttribute");
    for (int per_sm = D <= 128 ? 2 : 1; per_sm >= 1; --per_sm) {
      const int budget =
          std::min(optin, static_cast<int>(prop.sharedMemPerMultiprocessor) / per_sm - 1024);
      // Two 128-row stages: at D <= 128 that is what two CTAs' shares of
      // shared memory hold; at D = 256 a third 64 KB stage left no room for
      // the normalise kernel's CTAs to start next to the score kernel's, and
      // measured slower (MQA-style call 27.2 us against 26.0 with two).
      for (p->stages = kQkStreamStages; p->stages >= 2; --p->stages) {
        p->b_off = p->stages * p->stage_bytes;
        p->red_off = p->b_off + 2 * 2 * p->npad * D * 2;
        p->bar_off = p->red_off + kMmaAccWarps * p->npad * 8;
        p->lens_off = p->bar_off + (2 * kMaxStages + 10) * 8 + 32;
        p->q_off = 0;
        p->smem = p->lens_off + (B + 1) * 4 + 1024;
        if (p->smem <= budget || p->stages == 2) break;
      }
      // CTAs an SM: the occupancy query, or where it gives fewer, what the
      // SM's shared memory, registers and threads hold. (For this kernel the
      // query answered one CTA an SM at every shared-memory size, where two
      // of 84 KB ran side by side and 20 % faster. The CTAs do not wait on
      // one another, so a count that were too high would only make a second
      // wave.)
      int occ = 0;
      e2 = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                std::min(p->smem, optin));
      if (e2 != cudaSuccess) return qfail_cuda(e2, "cudaFuncSetAttribute");
      e2 = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kfn, p->threads, p->smem);
      if (e2 != cudaSuccess) return qfail_cuda(e2, "occupancy query");
      if (occ < per_sm)
        occ = std::max(occ, resident_ctas(reinterpret_cast<const void*>(kfn), p->threads, p->smem, prop));
      if (occ >= per_sm || per_sm == 1) {
        p->split_units = p->hgroups * std::max(1, sms * per_sm / p->hgroups);
        break;
      }
    }
    p->rows_per_split = p->R;
    p->nsplit = 1;
    if (p->smem > optin && auto_stream) {
      // Too large a query operand to double-buffer next to two stages (64
      // heads at D = 256): the fixed-split kernel, which keeps one.
      p->engine = kQkEngineTensor;
      p->threads = kQkMmaThreads;
      goto fixed_splits;
    }
    if (p->smem > optin)
      return qfail(GQA_AV_ERR_UNSUPPORTED, "plan needs %d B of shared memory (limit %d)", p->smem,
                   optin);
    // Partial pairs: two slots a CTA; then one slot per tile held whole.
    p->whole_off = static_cast<size_t>(2) * p->split_units * p->heads * sizeof(float2);
    p->ws_bytes = p->whole_off + static_cast<size_t>(p->tiles) * p->heads * sizeof(float2);
    norm_layout(p, B, Cmax, Hq, sms);
    if (static_cast<long long>(B) * p->norm_ctas_per_b > 0x7fffffffLL)
      return qfail(GQA_AV_ERR_UNSUPPORTED, "normalise grid too large");
    return GQA_AV_OK;
  }
fixed_splits:
  // FMA kernel: one CTA per SM on few-tile shapes. Tensor-core kernel: on
  // short streams with D <= 128 (at most 2048 rows a CTA at two CTAs per SM),
  // about two CTAs per SM with a ring of about 96 KiB; otherwise, like the FMA
  // kernel, a deep ring of about 160 KiB and one CTA per SM (each measured
  // faster in its regime).
  const long long tile_rows = static_cast<long long>(p->tiles) * Cmax;
  const bool short_tc = tensor && D <= 128 && tile_rows <= 2048LL * 2 * sms;
  // Short streams: at most two CTAs per SM in all, so that every split is
  // resident from the start (rounding up made a 32-tile ragged batch 320 CTAs
  // for 304 slots, and the 16 that waited for a slot added a second wave).
  long long want = short_tc ? std::max(1, 2 * sms / p->tiles)
                   : p->tiles < sms ? std::max(1, sms / p->tiles)
                                    : (2LL * sms + p->tiles - 1) / p->tiles;
  want = std::max<long long>(1, std::min<long long>(want, (Cmax + p->R - 1) / p->R));
  const int rps0 = static_cast<int>((Cmax + want - 1) / want);
  p->rows_per_split = (rps0 + p->R - 1) / p->R * p->R;
  p->nsplit = (Cmax + p->rows_per_split - 1) / p->rows_per_split;
  if (static_cast<long long>(p->tiles) * p->nsplit > 0x7fffffffLL)
    return qfail(GQA_AV_ERR_UNSUPPORTED, "grid too large");

  const int q_bytes = p->heads * D * 4;
  // FMA kernel: 3 stages (2 if that does not fit). Tensor-core kernel: a stage
  // per 128 rows of the split, as many as the ring above holds (2 to 8).
  const int iters = p->rows_per_split / p->R;
  const int ring = short_tc ? 98304 : 163840;
  const int want_stages =
      tensor ? std::max(2, std::min(std::min(kMaxStages, iters), ring / p->stage_bytes)) : 3;
  for (p->stages = want_stages; p->stages >= 2; --p->stages) {
    if (tensor) {
      p->b_off = p->stages * p->stage_bytes;
      p->red_off = p->b_off + 2 * p->npad * D * 2;
      p->bar_off = p->red_off + kMmaAccWarps * p->npad * 8;
      p->q_off = 0;
      p->smem = p->bar_off + (2 * kMaxStages + 6) * 8 + 8 + 1024;
    } else {
      p->q_off = p->stages * p->stage_bytes;
      p->red_off = p->q_off + (q_bytes + 127) / 128 * 128;
      p->bar_off = p->red_off + kQkConsumerWarps * 16 * 8;
      p->b_off = 0;
      p->smem = p->bar_off + 2 * kMaxStages * 8 + 1024;  // + alignment slack
    }
    if (p->smem <= optin) break;
  }
  if (p->smem > optin)
    return qfail(GQA_AV_ERR_UNSUPPORTED, "plan needs %d B of shared memory (limit %d)", p->smem,
                 optin);
  p->ws_bytes = static_cast<size_t>(p->tiles) * p->nsplit * p->heads * sizeof(float2);

  // Normalise: about kQkNormBatch scores a thread, so each thread has one
  // round of loads in flight.
  norm_layout(p, B, Cmax, Hq, sms);
  if (static_cast<long long>(B) * p->norm_ctas_per_b > 0x7fffffffLL)
    return qfail(GQA_AV_ERR_UNSUPPORTED, "normalise grid too large");
  return GQA_AV_OK;
}

struct Ws {
  void* base = nullptr;
  size_t bytes = 0;
};
std::map<int, Ws> g_qk_ws;

int workspace(int dev, size_t need, cudaStream_t stream, Ws* out) {
  std::lock_guard<std::mutex> lk(g_qk_mu);
  Ws& w = g_qk_ws[dev];
  if (w.base && w.bytes >= need) {
    *out = w;
    return GQA_AV_OK;
  }
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(stream, &cs);
  if (e != cudaSuccess) return qfail_cuda(e, "cudaStreamIsCapturing");
  if (cs != cudaStreamCaptureStatusNone)
    return qfail(GQA_AV_ERR_NOMEM,
                 "workspace must grow to %zu B but the stream is capturing; make one call with "
                 "the largest shape before capture",
                 need);
  const size_t bytes = std::max(need, w.bytes + w.bytes / 2);
  if (w.base) {
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return qfail_cuda(e, "cudaDeviceSynchronize");
    cudaFree(w.base);
    w.base = nullptr;
    w.bytes = 0;
  }
  void* p = nullptr;
  e = cudaMalloc(&p, bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return qfail(GQA_AV_ERR_NOMEM, "cudaMalloc(%zu) failed: %s", bytes, cudaGetErrorString(e));
  }
  e = cudaMemset(p, 0, kQkHeaderBytes);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    cudaFree(p);
    return qfail_cuda(e, "zeroing the workspace header");
  }
  w.base = p;
  w.bytes = bytes;
  *out = w;
  return GQA_AV_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 g_qk_encode = nullptr;

// K viewed as 4-D {D, Hkv, Cmax, B} (innermost first); box {64, 1, R, 1} in
// the 128-byte swizzle (one 128-byte line per row and part).
int encode_k_map(CUtensorMap* m, const void* k, int B, int Cmax, int Hkv, int D, int R) {
  {
    std::lock_guard<std::mutex> lk(g_qk_mu);
    if (!g_qk_encode) {
      void* f = nullptr;
      cudaDriverEntryPointQueryResult q;
      cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                                       cudaEnableDefault, &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !f)
        return qfail(GQA_AV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
      g_qk_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
  }
  const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)Cmax, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)Hkv * D * 2,
                                 (cuuint64_t)Cmax * Hkv * D * 2};
  const cuuint32_t box[4] = {64, 1, (cuuint32_t)R, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = g_qk_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, const_cast<void*>(k), dims,
                           strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return qfail(GQA_AV_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled (K) failed (%d)", (int)r);
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

extern "C" int gqa_qk_softmax_decode_tuned(const float* q, const void* k_cache,
                                           const int32_t* seq_lens, float* attn, int B, int Cmax,
                                           int Hq, int Hkv, int D, int k_dtype, float scale,
                                           int mode, int engine, void* stream_) {
  g_qk_error.clear();
  if (!q || !k_cache || !attn)
    return qfail(GQA_AV_ERR_INVALID, "q, k_cache and attn must be non-NULL");
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_cache) |
       reinterpret_cast<uintptr_t>(attn)) & 15u)
    return qfail(GQA_AV_ERR_UNSUPPORTED, "q, k_cache and attn must be 16-byte aligned");
  int rc = check_args(B, Cmax, Hq, Hkv, D, k_dtype, mode);
  if (rc) return rc;
  const int G = Hq / Hkv;
  const int heads = (mode == GQA_AV_MODE_GQA || (mode == GQA_AV_MODE_AUTO && G > 1)) ? G : 1;
  if (heads > kQkMaxHeads)
    return qfail(GQA_AV_ERR_UNSUPPORTED, "%d heads per KV head, at most %d", heads, kQkMaxHeads);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return qfail_cuda(e, "cudaGetDevice");
  QkPlan pl{};
  if ((rc = plan(dev, B, Cmax, Hq, Hkv, D, k_dtype, mode, engine, &pl))) return rc;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  Ws ws;
  if ((rc = workspace(dev, kQkHeaderBytes + pl.ws_bytes, stream, &ws))) return rc;

  QkParams p;
  if ((rc = encode_k_map(&p.k_map, k_cache, B, Cmax, Hkv, D, pl.R))) return rc;
  p.q = q;
  p.seq_lens = seq_lens;
  p.attn = attn;
  p.status = static_cast<unsigned int*>(ws.base);
  p.stats = reinterpret_cast<float2*>(static_cast<char*>(ws.base) + kQkHeaderBytes);
  p.scale = scale;
  p.B = B; p.Cmax = Cmax; p.Hq = Hq; p.Hkv = Hkv; p.D = D; p.G = Hq / Hkv;
  p.heads = pl.heads; p.hgroups = pl.hgroups; p.nc = pl.nc; p.rs = pl.rs; p.R = pl.R;
  p.stages = pl.stages; p.rows_per_split = pl.rows_per_split; p.nsplit = pl.nsplit;
  p.parts = pl.parts; p.stage_bytes = static_cast<uint32_t>(pl.stage_bytes);
  p.q_off = pl.q_off; p.red_off = pl.red_off; p.bar_off = pl.bar_off;
  p.timeout_ns = kQkTimeoutNs;
  p.b_off = pl.b_off;
  p.tmem_cols = static_cast<uint32_t>(pl.tmem_cols);
  p.split_units = pl.split_units;
  p.lens_off = static_cast<uint32_t>(pl.lens_off);
  p.stats_whole = reinterpret_cast<float2*>(static_cast<char*>(ws.base) + kQkHeaderBytes +
                                            pl.whole_off);

  QkKernel k;
  if (pl.engine == kQkEngineStream)
    k = k_dtype == GQA_AV_BF16 ? pick_stream<Bf16Tag>(pl.npad / 16) : pick_stream<Fp16Tag>(pl.npad / 16);
  else if (pl.engine == kQkEngineTensor)
    k = k_dtype == GQA_AV_BF16 ? pick_mma<Bf16Tag>(pl.npad / 16) : pick_mma<Fp16Tag>(pl.npad / 16);
  else
    k = k_dtype == GQA_AV_BF16 ? pick<Bf16Tag>(pl.gc) : pick<Fp16Tag>(pl.gc);
  if (!k) return qfail(GQA_AV_ERR_UNSUPPORTED, "no score kernel for this head count");
  e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, pl.smem);
  if (e != cudaSuccess) return qfail_cuda(e, "cudaFuncSetAttribute");
  void* args1[] = {&p};
  const unsigned grid1 = pl.engine == kQkEngineStream ? static_cast<unsigned>(pl.split_units)
                                                      : static_cast<unsigned>(pl.tiles * pl.nsplit);
  e = launch_pdl(reinterpret_cast<const void*>(k), dim3(grid1), dim3(pl.threads), pl.smem, stream,
                 args1);
  if (e != cudaSuccess) return qfail_cuda(e, "score kernel launch");

  QkNormParams n;
  n.stats = p.stats;
  n.seq_lens = seq_lens;
  n.attn = attn;
  n.B = B; n.Cmax = Cmax; n.Hq = Hq; n.heads = pl.heads; n.hgroups = pl.hgroups;
  n.rows_per_split = pl.rows_per_split; n.nsplit = pl.nsplit;
  n.rows_per_cta = pl.norm_rows; n.ctas_per_b = pl.norm_ctas_per_b;
  n.split_units = pl.split_units;
  n.stats_whole = p.stats_whole;
  void* args2[] = {&n};
  e = launch_pdl(pl.engine == kQkEngineStream
                     ? reinterpret_cast<const void*>(gqa_qk_stream_normalize)
                     : reinterpret_cast<const void*>(gqa_qk_normalize_kernel),
                 dim3(B * pl.norm_ctas_per_b), dim3(kQkNormThreads), 0, stream, args2);
  if (e != cudaSuccess) return qfail_cuda(e, "normalise kernel launch");
  return GQA_AV_OK;
}

extern "C" int gqa_qk_softmax_decode(const float* q, const void* k_cache, const int32_t* seq_lens,
                                     float* attn, int B, int Cmax, int Hq, int Hkv, int D,
                                     int k_dtype, float scale, int mode, void* stream) {
  return gqa_qk_softmax_decode_tuned(q, k_cache, seq_lens, attn, B, Cmax, Hq, Hkv, D, k_dtype,
                                     scale, mode, 0, stream);
}

extern "C" int gqa_qk_device_status(void* stream_, int clear) {
  g_qk_error.clear();
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return qfail_cuda(e, "cudaGetDevice");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return qfail_cuda(e, "cudaStreamSynchronize");
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_qk_mu);
    auto it = g_qk_ws.find(dev);
    if (it != g_qk_ws.end()) base = it->second.base;
  }
  if (!base) return GQA_AV_OK;
  unsigned word = 0;
  e = cudaMemcpy(&word, base, sizeof word, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return qfail_cuda(e, "reading the status word");
  if (word && clear) {
    e = cudaMemset(base, 0, sizeof word);
    if (e != cudaSuccess) return qfail_cuda(e, "clearing the status word");
  }
  if (word)
    return qfail(GQA_AV_ERR_DEVICE_TIMEOUT, "a bounded wait in the score kernel ran out (0x%x)",
                 word);
  return GQA_AV_OK;
}

extern "C" const char* gqa_qk_last_error(void) { return g_qk_error.c_str(); }
