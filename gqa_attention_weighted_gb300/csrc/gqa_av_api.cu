// Host side of the C ABI declared in include/gqa_av.h: argument checks, mode
// resolution (the override knob on the page "pytorch/executorch pull 21063",
// bullet on `gqa_override`), launch planning, the per-device workspace, TMA
// tensor-map encoding and dispatch to the kernel instantiations.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <numeric>
#include <string>
#include <tuple>

#include "gqa_av.h"
#define GQA_AV_COMBINE_KERNEL  // the split combine kernel lives in this translation unit
#include "gqa_av_generic.cuh"
#include "gqa_av_kernel.cuh"
#include "gqa_av_mma.cuh"
#include "gqa_av_stream.cuh"

namespace gqa_av {

// Explicit instantiations live in gqa_av_bf16.cu / gqa_av_fp16.cu.
#define GQA_AV_DECLARE(TAG, GC)                                                          \
  extern template cudaError_t launch<TAG, GC>(const Params&, int, int, cudaStream_t);    \
  extern template cudaError_t occupancy<TAG, GC>(int, int, int*);
#define GQA_AV_DECLARE_ALL(TAG)                                                              \
  GQA_AV_DECLARE(TAG, 1) GQA_AV_DECLARE(TAG, 2) GQA_AV_DECLARE(TAG, 3) GQA_AV_DECLARE(TAG, 4) \
  GQA_AV_DECLARE(TAG, 5) GQA_AV_DECLARE(TAG, 6) GQA_AV_DECLARE(TAG, 7) GQA_AV_DECLARE(TAG, 8) \
  GQA_AV_DECLARE(TAG, 12)
GQA_AV_DECLARE_ALL(Bf16Tag)
GQA_AV_DECLARE_ALL(Fp16Tag)
#define GQA_AV_DECLARE_MMA(TAG, NB)                                                      \
  extern template cudaError_t launch_mma<TAG, NB>(const Params&, int, int, cudaStream_t); \
  extern template cudaError_t occupancy_mma<TAG, NB>(int, int, int*);
#define GQA_AV_DECLARE_MMA_ALL(TAG) \
  GQA_AV_DECLARE_MMA(TAG, 1) GQA_AV_DECLARE_MMA(TAG, 2) GQA_AV_DECLARE_MMA(TAG, 3) GQA_AV_DECLARE_MMA(TAG, 4)
GQA_AV_DECLARE_MMA_ALL(Bf16Tag)
GQA_AV_DECLARE_MMA_ALL(Fp16Tag)
#define GQA_AV_DECLARE_STREAM(TAG, NB)                                                      \
  extern template cudaError_t launch_stream<TAG, NB>(const Params&, int, int, cudaStream_t); \
  extern template cudaError_t occupancy_stream<TAG, NB>(int, int, int*);
#define GQA_AV_DECLARE_STREAM_ALL(TAG)                                                    \
  GQA_AV_DECLARE_STREAM(TAG, 1) GQA_AV_DECLARE_STREAM(TAG, 2) GQA_AV_DECLARE_STREAM(TAG, 3) \
  GQA_AV_DECLARE_STREAM(TAG, 4)
GQA_AV_DECLARE_STREAM_ALL(Bf16Tag)
GQA_AV_DECLARE_STREAM_ALL(Fp16Tag)

namespace {

// Heads per thread; 16 would exceed the registers a 9-warp CTA can give a thread.
constexpr int kHeadChunks[] = {12, 8, 7, 6, 5, 4, 3, 2, 1};
constexpr size_t kHeaderBytes = 256;               // device status word + padding
constexpr long long kWaitTimeoutNs = 2000000000LL; // 2 s bound on every mbarrier wait

thread_local std::string g_last_error;

int fail(int status, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return status;
}

int fail_cuda(cudaError_t e, const char* what) {
  return fail(GQA_AV_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ----------------------------------------------------------------- dispatch
using LaunchFn = cudaError_t (*)(const Params&, int, int, cudaStream_t);
using OccFn = cudaError_t (*)(int, int, int*);
struct Kernel {
  LaunchFn launch;
  OccFn occupancy;
};

constexpr int kEngineFma = 1;     // CUDA-core packed-FMA kernel
constexpr int kEngineTensor = 2;  // tcgen05 tensor-core kernel
constexpr int kEngineGeneric = 3; // any D, element-aligned pointers (plain loads)
constexpr int kMaxMmaHeads = 64;  // N <= 64: B ring and tensor memory stay small

template <typename Tag>
bool pick_mma(int nb, Kernel* k) {
  switch (nb) {
    case 1: *k = {launch_mma<Tag, 1>, occupancy_mma<Tag, 1>}; return true;
    case 2: *k = {launch_mma<Tag, 2>, occupancy_mma<Tag, 2>}; return true;
    case 3: *k = {launch_mma<Tag, 3>, occupancy_mma<Tag, 3>}; return true;
    case 4: *k = {launch_mma<Tag, 4>, occupancy_mma<Tag, 4>}; return true;
    default: return false;
  }
}

template <typename Tag>
bool pick_stream(int nb, Kernel* k) {
  switch (nb) {
    case 1: *k = {launch_stream<Tag, 1>, occupancy_stream<Tag, 1>}; return true;
    case 2: *k = {launch_stream<Tag, 2>, occupancy_stream<Tag, 2>}; return true;
    case 3: *k = {launch_stream<Tag, 3>, occupancy_stream<Tag, 3>}; return true;
    case 4: *k = {launch_stream<Tag, 4>, occupancy_stream<Tag, 4>}; return true;
    default: return false;
  }
}

template <typename Tag>
bool pick(int gc, Kernel* k) {
  switch (gc) {
#define GQA_AV_CASE(GC)                          \
  case GC:                                       \
    *k = {launch<Tag, GC>, occupancy<Tag, GC>};  \
    return true;
    GQA_AV_CASE(1) GQA_AV_CASE(2) GQA_AV_CASE(3) GQA_AV_CASE(4) GQA_AV_CASE(5)
    GQA_AV_CASE(6) GQA_AV_CASE(7) GQA_AV_CASE(8) GQA_AV_CASE(12)
#undef GQA_AV_CASE
    default:
      return false;
  }
}

// `sel` is the head chunk (FMA kernel) or N / 16 (tensor-core kernels);
// kEngineStream is the streamed tensor-core kernel.
constexpr int kEngineStream = 4;

bool pick_kernel(int v_dtype, int engine, int sel, Kernel* k) {
  if (engine == kEngineStream)
    return v_dtype == GQA_AV_BF16 ? pick_stream<Bf16Tag>(sel, k) : pick_stream<Fp16Tag>(sel, k);
  if (engine == kEngineTensor)
    return v_dtype == GQA_AV_BF16 ? pick_mma<Bf16Tag>(sel, k) : pick_mma<Fp16Tag>(sel, k);
  return v_dtype == GQA_AV_BF16 ? pick<Bf16Tag>(sel, k) : pick<Fp16Tag>(sel, k);
}

// ------------------------------------------------------------- device info
struct DeviceInfo {
  int sms = 0;
  int smem_optin = 0;
  int smem_per_sm = 0;
  bool ok = false;
};

std::mutex g_mu;
std::map<int, DeviceInfo> g_devices;
std::map<std::tuple<int, int, int, int, int>, int> g_occupancy;  // (dev, dtype, engine, sel, smem)

int device_info(int dev, DeviceInfo* out) {
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_devices.find(dev);
  if (it != g_devices.end()) {
    *out = it->second;
    return GQA_AV_OK;
  }
  DeviceInfo di;
  cudaError_t e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&di.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&di.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaDeviceGetAttribute");
  di.ok = true;
  g_devices[dev] = di;
  *out = di;
  return GQA_AV_OK;
}

int ctas_per_sm(int dev, int smem_limit, int v_dtype, int engine, int sel, int smem, int* n) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_occupancy.find(std::make_tuple(dev, v_dtype, engine, sel, smem));
    if (it != g_occupancy.end()) {
      *n = it->second;
      return GQA_AV_OK;
    }
  }
  Kernel kern;
  if (!pick_kernel(v_dtype, engine, sel, &kern))
    return fail(GQA_AV_ERR_UNSUPPORTED, "no kernel for engine %d / %d", engine, sel);
  int k = 0;
  cudaError_t e = kern.occupancy(smem_limit, smem, &k);
  if (e != cudaSuccess) return fail_cuda(e, "occupancy query");
  std::lock_guard<std::mutex> lk(g_mu);
  g_occupancy[std::make_tuple(dev, v_dtype, engine, sel, smem)] = k;
  *n = k;
  return GQA_AV_OK;
}

// ------------------------------------------------------------------- plan
struct Plan {
  int mode, heads, gc, nc, dt, ndt, ct, row_par, R, stages, nsplit, rows_per_split;
  int hgroups, tiles, ap, avec, smem, occ;
  int parts, cols_per_cta, ctas_per_tile;  // split combine launch (combine set)
  int combine;                             // the split combine runs after the main kernel
  int grid;                                // CTAs of the main kernel
  int split_units;                         // tensor core: CTAs the context is balanced over
  int balanced;                            // tensor core: splits balanced over the batch's lengths
  int stream;                              // tensor core: the streamed kernel (split_mode 3)
  uint32_t lens_off;                       // streamed kernel: shared-memory offset of the lengths
  int chunk_rows;                          // rows per V box (R, or a paged block)
  int one_per_sm;                          // shared memory padded so one CTA fits per SM
  int early;                               // stages issued before the length is read
  int engine;                              // kEngineFma or kEngineTensor
  int nmma;                                // tensor core: N (heads padded to 16)
  int v_halves;                            // tensor core: 64-column V boxes per stage
  int tmem_cols;                           // tensor core: tensor-memory columns
  int cvt_warps;                           // tensor core: weight-conversion warps
  uint32_t b_off;                          // tensor core: B ring offset
  int attn_tma;                            // attn weights by TMA (rows of Hq % 4 == 0 floats)
  uint32_t v_stage_bytes, a_off, bar_off;
  size_t ws_bytes;  // partials only
};

int check_shape_any_d(int B, int Cmax, int Hq, int Hkv, int D, int v_dtype, int mode);

int check_shape(int B, int Cmax, int Hq, int Hkv, int D, int v_dtype, int mode) {
  int rc = check_shape_any_d(B, Cmax, Hq, Hkv, D, v_dtype, mode);
  if (rc) return rc;
  if (D % 8 != 0) return fail(GQA_AV_ERR_UNSUPPORTED, "D=%d is not a multiple of 8", D);
  return GQA_AV_OK;
}

// The checks that hold for every kernel, the generic one included.
int check_shape_any_d(int B, int Cmax, int Hq, int Hkv, int D, int v_dtype, int mode) {
  if (B <= 0 || Cmax <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0)
    return fail(GQA_AV_ERR_INVALID, "sizes must be positive (B=%d Cmax=%d Hq=%d Hkv=%d D=%d)", B,
                Cmax, Hq, Hkv, D);
  if (Hq % Hkv != 0)
    return fail(GQA_AV_ERR_INVALID, "Hq=%d is not a multiple of Hkv=%d", Hq, Hkv);
  if (v_dtype != GQA_AV_BF16 && v_dtype != GQA_AV_FP16)
    return fail(GQA_AV_ERR_INVALID, "unknown v_dtype %d", v_dtype);
  if (mode != GQA_AV_MODE_AUTO && mode != GQA_AV_MODE_PER_HEAD && mode != GQA_AV_MODE_GQA)
    return fail(GQA_AV_ERR_INVALID, "unknown mode %d", mode);
  return GQA_AV_OK;
}

// Kernel instantiation of a plan: head chunk (FMA) or N / 16 (tensor core).
int kernel_sel(const Plan& p) { return p.engine == kEngineTensor ? p.nmma / 16 : p.gc; }

// The engine code of the kernel that runs a plan (the streamed kernel is a
// schedule of the tensor-core engine).
int kernel_engine(const Plan& p) { return p.stream ? kEngineStream : p.engine; }

// Shared memory of a tensor-core plan, from a 1024-byte-aligned base (1 KiB of
// slack lets the kernel align the dynamic allocation): [V ring, stages x R x
// 256 B] [attn ring] [B ring, stages x (hi, lo) x N x R x 2 B] [mbarriers,
// tensor-memory address, flag].
void layout_mma(Plan* p, int min_smem) {
  p->v_stage_bytes = static_cast<uint32_t>(p->R) * 256;
  const size_t vring = static_cast<size_t>(p->stages) * p->v_stage_bytes;
  p->a_off = static_cast<uint32_t>(align_up(vring, 128));
  const size_t aring = static_cast<size_t>(p->stages) * p->R * p->ap * 4;
  p->b_off = static_cast<uint32_t>(align_up(p->a_off + aring, 128));
  const size_t bring = static_cast<size_t>(p->stages) * 2 * p->nmma * p->R * 2;
  p->bar_off = static_cast<uint32_t>(align_up(p->b_off + bring, 16));
  const size_t bars = (3 * kMaxStages + 5) * 8 + 8 + 48;  // + the CTA's split record (9 ints)
  p->smem = std::max(static_cast<int>(p->bar_off + bars + 1024), min_smem);
}

// Shared memory of a plan: [V ring | reduction buffer] [attn ring] [mbarriers] [flag].
void layout(Plan* p, int min_smem = 0) {
  p->v_stage_bytes = static_cast<uint32_t>(p->R) * p->dt * 2;
  const size_t vring = static_cast<size_t>(p->stages) * p->v_stage_bytes;
  const size_t red = static_cast<size_t>(p->row_par) * p->heads * p->dt * 4;
  p->a_off = static_cast<uint32_t>(align_up(std::max(vring, red), 128));
  const size_t aring = static_cast<size_t>(p->stages) * p->R * p->ap * 4;
  p->bar_off = static_cast<uint32_t>(align_up(p->a_off + aring, 16));
  p->smem = std::max(static_cast<int>(p->bar_off + 2 * kMaxStages * 8 + 16), min_smem);
}

// attn weights of a stage. By TMA when attn rows are 16-byte multiples
// (Hq % 4 == 0): the box starts at the 4-aligned head at or below the CTA's
// first head (a TMA box must start 16-byte aligned) and is wide enough for
// every CTA's heads; otherwise by cp.async, `avec` floats a copy.
void attn_layout(Plan* p, int Hq) {
  const int max_off = p->heads % 4 == 0 ? 0 : (p->heads % 2 == 0 ? 2 : 3);
  const int aw = static_cast<int>(align_up(p->heads + max_off, 4));
  p->attn_tma = Hq % 4 == 0 && aw <= 256;
  p->ap = p->attn_tma ? aw : static_cast<int>(align_up(p->heads, 4));
  p->avec = 1;
  if (Hq % 4 == 0 && p->heads % 4 == 0) p->avec = 4;
  else if (Hq % 2 == 0 && p->heads % 2 == 0) p->avec = 2;
}

// Split-combine launch shape: `parts` threads per float4 column (a power of
// two <= 16), as many as keep its grid within about one CTA per SM. Its CTAs
// are small enough to start next to the main kernel's while that runs, so
// they are all waiting when the partials are complete (measured faster than
// a grid that only starts as the main kernel's CTAs leave).
// `slots`: the mean number of partials of one tile when known at plan time
// (streamed splits), else 0; `parts` is raised until one batch of a thread's
// loads covers them (an MQA-shaped call with about 20 partials a tile
// combined 0.7 us faster with 4 threads a column than with 2).
void combine_layout(Plan* p, int sms, long long slots = 0) {
  const int ncol4 = p->heads * p->dt / 4;
  const long long cols = static_cast<long long>(p->tiles) * ncol4;
  p->parts = 1;
  while (p->parts < 16 && (p->balanced || p->stream || p->parts < p->nsplit) &&
         cols * p->parts * 2 <= static_cast<long long>(sms) * kCombineThreads)
    p->parts *= 2;
  while (p->parts < 16 && slots > static_cast<long long>(kCombineBatch) * p->parts) p->parts *= 2;
  p->cols_per_cta = kCombineThreads / p->parts;
  p->ctas_per_tile = (ncol4 + p->cols_per_cta - 1) / p->cols_per_cta;
}

// The streamed tensor-core kernel (split_mode 3): about SMs x ctas_per_sm
// persistent CTAs (tuning nsplit: CTAs per SM, 1 to 4; default 2) in groups
// of one CTA per tile of a sequence, each CTA taking an equal run of its tile
// column's R-row stages (tuning rows_per_stage, a multiple of 16; default 64)
// through a ring of `stages` slots (default: as many as fit the CTA's share
// of the SM's shared memory, 2 to 8).
int plan_stream(Plan* p, const gqa_av_tuning* t, const DeviceInfo& di, int B, int Cmax, int dev,
                int v_dtype, int Hq) {
  const int per_sm = t && t->nsplit > 0 ? t->nsplit : 2;
  if (per_sm > 4) return fail(GQA_AV_ERR_INVALID, "streamed splits: nsplit=%d CTAs per SM, at most 4", per_sm);
  p->stream = 1;
  p->balanced = 0;
  p->early = 0;
  p->cvt_warps = 4;  // one CTA streams for the whole call: the widest conversion
  if (t && t->rows_per_stage > 0) {
    if (t->rows_per_stage % 16 || t->rows_per_stage > 256)
      return fail(GQA_AV_ERR_INVALID, "rows_per_stage=%d must be a multiple of 16, <= 256",
                  t->rows_per_stage);
    p->R = t->rows_per_stage;
  } else {
    // 64-row stages on shapes with at least as many tiles as SMs, 96-row
    // stages on the others (each measured faster in its regime).
    p->R = static_cast<long long>(B) * p->hgroups * p->ndt >= di.sms ? 64 : 96;
  }
  p->chunk_rows = p->R;
  p->rows_per_split = p->R;
  // K CTAs a group, one per tile of a sequence; as many groups as fit
  // per_sm CTAs on every SM (at least one).
  const int K = p->hgroups * p->ndt;
  p->split_units = K * std::max(1, di.sms * per_sm / K);
  p->grid = p->split_units;
  p->nsplit = per_sm;
  p->combine = 1;
  attn_layout(p, Hq);
  const int budget = std::min(di.smem_optin, di.smem_per_sm / per_sm - 1024);
  auto lay = [&] {
    layout_mma(p, 0);
    p->lens_off = static_cast<uint32_t>(align_up(p->smem - 1024, 16));
    p->smem = static_cast<int>(p->lens_off + (B + 1) * 4 + 1024);
  };
  if (t && t->stages > 0) {
    if (t->stages < 2 || t->stages > kMaxStages)
      return fail(GQA_AV_ERR_INVALID, "stages=%d must be in [2, %d]", t->stages, kMaxStages);
    p->stages = t->stages;
    lay();
  } else {
    // About 64 KiB of V in flight a CTA (4 stages of 64 rows, 3 of 96 or
    // more, 2 of 128 or more), fewer if the CTA's share of shared memory is
    // smaller, at least 2.
    const int pref = std::max(2, std::min(kMaxStages, 65536 / (p->R * 256) + (p->R == 96)));
    for (p->stages = pref; p->stages > 2; --p->stages) {
      lay();
      if (p->smem <= budget) break;
    }
    lay();
  }
  if (p->smem > di.smem_optin)
    return fail(GQA_AV_ERR_UNSUPPORTED, "plan needs %d B of shared memory (limit %d)", p->smem,
                di.smem_optin);
  if (t && t->early_stages > p->stages)
    return fail(GQA_AV_ERR_INVALID, "early_stages=%d must be in [1, stages=%d]", t->early_stages,
                p->stages);
  int rc;
  if ((rc = ctas_per_sm(dev, di.smem_optin, v_dtype, kEngineStream, p->nmma / 16, p->smem, &p->occ)))
    return rc;
  if (p->occ < 1) return fail(GQA_AV_ERR_UNSUPPORTED, "kernel does not fit on an SM");
  p->one_per_sm = 0;
  p->ws_bytes = static_cast<size_t>(2) * p->split_units * p->heads * p->dt * sizeof(float);
  // A tile's partials: about one per group over the B sequences of its
  // column, plus the cut at each end.
  combine_layout(p, di.sms, p->split_units / K / B + 2);
  (void)Cmax;
  return GQA_AV_OK;
}

int make_plan(int dev, int B, int Cmax, int Hq, int Hkv, int D, int v_dtype, int mode,
              const gqa_av_tuning* t, Plan* p, int block_size = 0) {
  int rc = check_shape(B, Cmax, Hq, Hkv, D, v_dtype, mode);
  if (rc) return rc;
  DeviceInfo di;
  if ((rc = device_info(dev, &di))) return rc;

  const int G = Hq / Hkv;
  p->mode = mode == GQA_AV_MODE_AUTO ? (G > 1 ? GQA_AV_MODE_GQA : GQA_AV_MODE_PER_HEAD) : mode;
  p->heads = p->mode == GQA_AV_MODE_GQA ? G : 1;
  p->hgroups = Hq / p->heads;
  p->gc = 1;
  for (int c : kHeadChunks)
    if (p->heads % c == 0) { p->gc = c; break; }
  p->nc = p->heads / p->gc;

  // Engine. The tensor-core kernel takes head groups of up to 64 heads and
  // D >= 64 that splits into 128-column tiles (D <= 128 or D % 128 == 0);
  // the packed-FMA kernel takes the rest, or any shape when asked for (a
  // dtile override also selects it). Where both apply the library picks by
  // what bounds the call (measured on GB300): 8 or more heads a CTA make the
  // FMA kernel's arithmetic the bound, and so do long streams (the FMA issue
  // rate falls behind HBM); short one-wave calls with few heads are bound by
  // latency, where the FMA kernel's lighter pipeline is faster.
  const bool mma_ok = p->heads <= kMaxMmaHeads && D >= 64 && (D <= kMmaM || D % kMmaM == 0);
  const int want_engine = t ? t->engine : 0;
  if (want_engine < 0 || want_engine > kEngineTensor)
    return fail(GQA_AV_ERR_INVALID, "engine=%d must be 0 (auto), 1 (FMA) or 2 (tensor)",
                want_engine);
  if (want_engine == kEngineTensor && !mma_ok)
    return fail(GQA_AV_ERR_UNSUPPORTED,
                "the tensor-core engine needs <= %d heads per CTA and D >= 64 with D <= 128 or "
                "D %% 128 == 0 (heads %d, D %d)",
                kMaxMmaHeads, p->heads, D);
  if (want_engine == kEngineTensor && t->dtile > 0 && t->dtile != std::min(D, kMmaM))
    return fail(GQA_AV_ERR_INVALID, "the tensor-core engine uses dtile = %d", std::min(D, kMmaM));
  const long long tile_rows =
      static_cast<long long>(B) * p->hgroups * Cmax * ((D + kMmaM - 1) / kMmaM);
  const bool prefer_tensor = p->heads >= 8 || tile_rows >= (1LL << 18);
  if (want_engine)
    p->engine = want_engine;
  else
    p->engine = mma_ok && !(t && t->dtile > 0) && prefer_tensor ? kEngineTensor : kEngineFma;
  const bool tensor = p->engine == kEngineTensor;

  if (tensor) {
    // One MMA covers 128 output columns; D <= 64 leaves the second half idle.
    // Two weight-conversion warps (8 warps, up to four CTAs an SM) where the
    // shape has fewer tiles than SMs, four (10 warps, two CTAs an SM) where
    // many long CTAs run in waves: each measured faster in its regime.
    p->cvt_warps = B * p->hgroups * ((D + kMmaM - 1) / kMmaM) < di.sms ? 2 : 4;
    p->dt = std::min(D, kMmaM);
    p->nmma = static_cast<int>(align_up(p->heads, 16));
    p->v_halves = p->dt > 64 ? 2 : 1;
    p->tmem_cols = 32;  // two D buffers of 2N columns (hi and lo products)
    while (p->tmem_cols < 4 * p->nmma) p->tmem_cols *= 2;
    p->row_par = 1;
  } else {
    // Output columns per CTA: a multiple of 8 dividing D, at most 256 (one TMA box).
    const int want_dt = (t && t->dtile > 0) ? t->dtile : 128;
    if (t && t->dtile > 0 && (t->dtile % 8 || D % t->dtile || t->dtile > 256))
      return fail(GQA_AV_ERR_INVALID, "dtile=%d must be a multiple of 8 dividing D=%d, <= 256",
                  t->dtile, D);
    p->dt = 0;
    for (int dt = std::min(want_dt, std::min(D, 256)); dt >= 8; dt -= 8)
      if (D % dt == 0 && (dt / 8) * p->nc <= 32 * consumer_warps(p->gc)) { p->dt = dt; break; }
    if (!p->dt)
      return fail(GQA_AV_ERR_UNSUPPORTED, "no column tile fits G=%d heads per CTA", p->heads);
    p->nmma = 0;
    p->v_halves = 0;
    p->tmem_cols = 0;
    p->cvt_warps = 0;
  }
  p->ndt = D / p->dt;
  p->ct = p->dt / 8;
  if (!tensor) p->row_par = 32 * consumer_warps(p->gc) / (p->ct * p->nc);

  // Context splits. With fewer tiles than SMs the grid is one wave of one CTA
  // per SM (shared memory is padded to more than half an SM so no SM takes
  // two); with many tiles it runs in waves (a split with no context exits at
  // once) and splits only balance ragged lengths.
  p->tiles = p->hgroups * B * p->ndt;
  // The tensor-core kernel keeps a small ring, so two of its CTAs share an
  // SM (measured: the occupancy query reports one, but per-SM traces show
  // two alive at once), and it pays a fixed cost per CTA: with few tiles it
  // is given about three times as many short splits as there are SMs, which
  // also balances ragged lengths (measured faster than one long split per SM).
  const bool few_tiles = !(t && t->nsplit > 0) && p->tiles < di.sms;
  const bool one_wave = few_tiles && !tensor;
  long long want;
  if (t && t->nsplit > 0) {
    want = t->nsplit;
  } else if (few_tiles && tensor) {
    want = (3LL * di.sms + p->tiles - 1) / p->tiles;
  } else if (one_wave) {
    want = di.sms / p->tiles;
  } else {
    const double v_bytes = static_cast<double>(B) * Cmax * (p->heads == 1 ? Hq : Hkv) * D * 2;
    const int waves = v_bytes > 256e6 ? 4 : 1;
    // Occupancy is not known yet: assume two CTAs per SM for the wave size.
    want = (2LL * di.sms * waves + p->tiles - 1) / p->tiles;
  }
  want = std::max<long long>(1, std::min<long long>(want, (Cmax + 7) / 8));
  const int rps0 = static_cast<int>((Cmax + want - 1) / want);

  // Rows per stage: about 32 KiB of V per stage (large boxes stream faster
  // per SM), a multiple of 8 rows (16, the MMA's K, for the tensor-core
  // kernel), dividing the split into equal stages.
  const int rq = tensor ? 16 : 8;
  int iters;
  if (t && t->rows_per_stage > 0) {
    if (t->rows_per_stage % rq || t->rows_per_stage > 256)
      return fail(GQA_AV_ERR_INVALID, "rows_per_stage=%d must be a multiple of %d, <= 256",
                  t->rows_per_stage, rq);
    p->R = t->rows_per_stage;
    iters = (rps0 + p->R - 1) / p->R;
  } else {
    // The tensor-core kernel runs faster the less shared memory a CTA holds
    // (measured: more CTAs stay resident, and the next call's CTAs start on an
    // SM while this call drains): 12 KiB of V per stage in a 3-stage ring, or
    // 16 KiB for the short splits of shapes with under 48 tiles (measured
    // faster there). 32 KiB for the FMA kernel.
    const int row_bytes = tensor ? 256 : 2 * p->dt;
    const int stage_bytes = tensor ? (few_tiles && p->tiles < 48 ? 16384 : 12288) : 32768;
    const int rmax = std::max(rq, std::min(256, stage_bytes / row_bytes) / rq * rq);
    iters = (rps0 + rmax - 1) / rmax;
    p->R = static_cast<int>(align_up((rps0 + iters - 1) / iters, rq));
  }
  p->chunk_rows = p->R;
  if (block_size > 0) {
    // Paged V: a stage is whole blocks (one box each) or a divisor of a block.
    if (p->R >= block_size) {
      const int unit = std::lcm(block_size, rq);
      if (unit > 256 || (t && t->rows_per_stage > 0 && p->R % unit))
        return fail(GQA_AV_ERR_INVALID, "rows_per_stage=%d does not fit blocks of %d rows",
                    p->R, block_size);
      p->R = std::max(unit, p->R / unit * unit);
      p->chunk_rows = block_size;
    } else {
      int r = p->R;
      while (r > rq && block_size % r) r -= rq;
      if (block_size % r || (t && t->rows_per_stage > 0 && r != p->R))
        return fail(GQA_AV_ERR_INVALID, "no stage of a multiple of %d rows divides blocks of %d",
                    rq, block_size);
      p->R = r;
      p->chunk_rows = r;
    }
    iters = (rps0 + p->R - 1) / p->R;
  }
  p->rows_per_split = p->R * iters;
  p->nsplit = (Cmax + p->rows_per_split - 1) / p->rows_per_split;
  // Splits of the tensor-core kernel on shapes that run in waves (as many
  // tiles as SMs or more): the context rows of the whole batch, read from
  // seq_lens, are spread evenly over tiles x nsplit CTAs, so ragged lengths
  // leave no CTA idle and every wave is full (measured 12% faster on the
  // ragged large-batch shape); rounding can give each sequence one split
  // more, so the grid has tiles more CTAs, and the split combine always runs.
  // With fewer tiles than SMs the grid is one wave and fixed splits are
  // faster: a CTA issues its first stage before it reads any length.
  const int want_split = t && t->split_mode > 0 ? t->split_mode : 0;
  if (want_split > 3)
    return fail(GQA_AV_ERR_INVALID,
                "split_mode=%d must be 0 (auto), 1 (fixed), 2 (balanced) or 3 (streamed)",
                want_split);
  if (want_split >= 2 && !tensor)
    return fail(GQA_AV_ERR_UNSUPPORTED, "balanced and streamed splits need the tensor-core engine");
  p->stream = 0;
  p->lens_off = 0;
  if (want_split == 3) {
    if (block_size > 0)
      return fail(GQA_AV_ERR_UNSUPPORTED, "streamed splits take a contiguous V cache");
    if (B > kStreamMaxB)
      return fail(GQA_AV_ERR_UNSUPPORTED, "streamed splits take at most %d sequences", kStreamMaxB);
    return plan_stream(p, t, di, B, Cmax, dev, v_dtype, Hq);
  }
  // The tensor-core engine streams by default (contiguous V, at most
  // kStreamMaxB sequences): measured faster than fixed or balanced splits on
  // every tensor-core workload (large batch 827 vs 882 us, its 1/8-context
  // twin 105 vs 117 us, MQA 19.5 vs 20.7 us, Phi 20.4 vs 21.3 us).
  if (want_split == 0 && tensor && block_size == 0 && B <= kStreamMaxB &&
      !(t && (t->nsplit > 0 || t->early_stages > 0)))
    return plan_stream(p, t, di, B, Cmax, dev, v_dtype, Hq);
  p->balanced = tensor && (want_split == 2 || (want_split == 0 && p->tiles >= di.sms));
  const long long grid =
      static_cast<long long>(p->tiles) * (p->balanced ? p->nsplit + 1 : p->nsplit);
  if (grid > 0x7fffffffLL) return fail(GQA_AV_ERR_UNSUPPORTED, "grid too large");
  p->grid = static_cast<int>(grid);
  p->split_units = p->balanced ? p->tiles * p->nsplit : 0;
  p->combine = p->balanced || p->nsplit > 1;

  if (t && t->stages > 0) {
    if (t->stages < 2 || t->stages > kMaxStages)
      return fail(GQA_AV_ERR_INVALID, "stages=%d must be in [2, %d]", t->stages, kMaxStages);
    p->stages = t->stages;
  } else {
    p->stages = std::max(2, std::min(3, iters));
  }
  attn_layout(p, Hq);
  p->one_per_sm = one_wave && static_cast<long long>(p->tiles) * p->nsplit <= di.sms;
  const int min_smem = p->one_per_sm ? di.smem_per_sm / 2 + 1024 : 0;
  auto lay = [&] { if (tensor) layout_mma(p, min_smem); else layout(p, min_smem); };
  lay();
  while (p->smem > di.smem_optin && p->stages > 2 && !(t && t->stages > 0)) {
    --p->stages;
    lay();
  }
  if (p->smem > di.smem_optin)
    return fail(GQA_AV_ERR_UNSUPPORTED, "plan needs %d B of shared memory (limit %d)", p->smem,
                di.smem_optin);
  // One stage goes out before the length is read: issuing the whole ring
  // early delays the first stage behind the others (measured slower on a
  // one-wave Llama-size grid), and a CTA past its length reads it for nothing.
  if (t && t->early_stages > 0) {
    if (t->early_stages > p->stages)
      return fail(GQA_AV_ERR_INVALID, "early_stages=%d must be in [1, stages=%d]",
                  t->early_stages, p->stages);
    p->early = t->early_stages;
  } else {
    p->early = 1;
  }
  // With balanced splits a CTA finds its split from the lengths, so it issues
  // nothing before it has read them.
  if (p->balanced) p->early = 0;

  if ((rc = ctas_per_sm(dev, di.smem_optin, v_dtype, kernel_engine(*p), kernel_sel(*p), p->smem,
                        &p->occ)))
    return rc;
  if (p->occ < 1) return fail(GQA_AV_ERR_UNSUPPORTED, "kernel does not fit on an SM");

  p->ws_bytes = p->combine
                    ? static_cast<size_t>(p->grid) * p->heads * p->dt * sizeof(float)
                    : 0;  // one partial slot a CTA
  combine_layout(p, di.sms);
  return GQA_AV_OK;
}

// Kernel parameters of one call of plan `pl` (everything but the tensor map).
void fill_params(Params* p, const Plan& pl, const float* attn, const int32_t* seq_lens,
                 float* out, void* status, void* partials, int B, int Cmax, int Hq, int Hkv,
                 int D) {
  p->attn = attn;
  p->seq_lens = seq_lens;
  p->out = out;
  p->status = static_cast<unsigned*>(status);
  p->ws = static_cast<float*>(partials);
  p->B = B; p->Cmax = Cmax; p->Hq = Hq; p->Hkv = Hkv; p->D = D; p->G = Hq / Hkv;
  p->heads = pl.heads; p->hgroups = pl.hgroups; p->dt = pl.dt; p->ndt = pl.ndt; p->ct = pl.ct;
  p->nc = pl.nc; p->row_par = pl.row_par; p->R = pl.R; p->stages = pl.stages;
  p->rows_per_split = pl.rows_per_split; p->nsplit = pl.nsplit;
  p->early_stages = pl.early;
  p->ap = pl.ap; p->avec = pl.avec; p->attn_tma = pl.attn_tma;
  p->a_stage_bytes = static_cast<uint32_t>(pl.R) * pl.ap * 4;
  p->v_stage_bytes = pl.v_stage_bytes; p->a_off = pl.a_off; p->bar_off = pl.bar_off;
  p->timeout_ns = kWaitTimeoutNs;
  p->full_wait_ns = kWaitTimeoutNs;
  p->withhold_last = 0;
  p->v_halves = pl.v_halves; p->b_off = pl.b_off; p->tmem_cols = static_cast<uint32_t>(pl.tmem_cols);
  p->cvt_warps = pl.cvt_warps;
  p->split_units = pl.split_units;
  p->balanced = pl.balanced;
  p->lens_off = pl.lens_off;
  p->chunk_rows = pl.chunk_rows;
  // attn is 16-byte aligned (checked before planning): a TMA source or a
  // cp.async of up to 16 bytes can start at any 4-head boundary of it.
}

// Launches the main kernel and, when the tile has several splits, the split
// combine right after it on the same stream.
cudaError_t launch_call(const Kernel& kern, const Plan& pl, const Params& p, cudaStream_t stream) {
  cudaError_t e = kern.launch(p, pl.grid, pl.smem, stream);
  if (e != cudaSuccess || !pl.combine) return e;
  CombineParams c;
  c.ws = p.ws;
  c.seq_lens = p.seq_lens;
  c.out = p.out;
  c.B = p.B; c.Cmax = p.Cmax; c.Hq = p.Hq; c.D = p.D;
  c.heads = pl.heads; c.dt = pl.dt; c.ndt = pl.ndt;
  c.rows_per_split = pl.rows_per_split; c.nsplit = pl.nsplit;
  c.tile_elems = pl.heads * pl.dt;
  c.parts = pl.parts; c.cols_per_cta = pl.cols_per_cta; c.ctas_per_tile = pl.ctas_per_tile;
  c.balanced = pl.stream ? kCombineStream : (pl.balanced ? kCombineBalanced : kCombineFixed);
  c.R = pl.R; c.hgroups = pl.hgroups; c.split_units = pl.split_units;
  return launch_combine(c, pl.tiles * pl.ctas_per_tile, stream);
}


// -------------------------------------------------------------- workspace
struct Workspace {
  void* base = nullptr;
  size_t bytes = 0;
  bool user = false;
};
std::map<int, Workspace> g_ws;
// Device -> status word of the no-allocation call's fixed array (registered
// by that call's per-device set-up).
std::map<int, void*> g_noalloc_status;

// Returns the workspace of `dev` with at least `need` bytes; grows outside capture.
int workspace(int dev, size_t need, cudaStream_t stream, Workspace* out) {
  std::lock_guard<std::mutex> lk(g_mu);
  Workspace& w = g_ws[dev];
  if (w.base && w.bytes >= need) {
    *out = w;
    return GQA_AV_OK;
  }
  if (w.user)
    return fail(GQA_AV_ERR_NOMEM, "caller workspace has %zu B, call needs %zu B", w.bytes, need);
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(stream, &cs);
  if (e != cudaSuccess) return fail_cuda(e, "cudaStreamIsCapturing");
  if (cs != cudaStreamCaptureStatusNone)
    return fail(GQA_AV_ERR_NOMEM,
                "workspace must grow to %zu B but the stream is capturing; make one call with "
                "the largest shape before capture",
                need);
  const size_t bytes = std::max(need, w.bytes + w.bytes / 2);
  if (w.base) {
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail_cuda(e, "cudaDeviceSynchronize");
    cudaFree(w.base);
    w.base = nullptr;
    w.bytes = 0;
  }
  void* p = nullptr;
  e = cudaMalloc(&p, bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(GQA_AV_ERR_NOMEM, "cudaMalloc(%zu) failed: %s", bytes, cudaGetErrorString(e));
  }
  e = cudaMemset(p, 0, kHeaderBytes);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    cudaFree(p);
    return fail_cuda(e, "zeroing the workspace header");
  }
  w.base = p;
  w.bytes = bytes;
  *out = w;
  return GQA_AV_OK;
}

// ------------------------------------------------------------ tensor maps
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int encode_fn(PFN_cuTensorMapEncodeTiled_v12000* fn) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_encode) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e =
        cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !f)
      return fail(GQA_AV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  *fn = g_encode;
  return GQA_AV_OK;
}

// V viewed as 4-D {D, Hkv, Cmax, B} (innermost first); box {dt, 1, R, 1}, or
// for the tensor-core kernel {64, 1, R, 1} with the 128-byte swizzle its A
// operand is read in.
// A paged cache is the same view of the block pool: {D, Hkv, block_size,
// num_blocks} with a box of `R` = chunk rows.
int encode_v_map(CUtensorMap* m, const void* v, int B, int Cmax, int Hkv, int D, int dt, int R,
                 bool mma) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  int rc = encode_fn(&enc);
  if (rc) return rc;
  const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)Cmax, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)Hkv * D * 2,
                                 (cuuint64_t)Cmax * Hkv * D * 2};
  const cuuint32_t box[4] = {(cuuint32_t)(mma ? 64 : dt), 1, (cuuint32_t)R, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, const_cast<void*>(v), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   mma ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(GQA_AV_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return GQA_AV_OK;
}

// attn viewed as 3-D {Hq, Cmax, B} (innermost first); box {width, R, 1}.
int encode_attn_map(CUtensorMap* m, const float* attn, int B, int Cmax, int Hq, int width, int R) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  int rc = encode_fn(&enc);
  if (rc) return rc;
  const cuuint64_t dims[3] = {(cuuint64_t)Hq, (cuuint64_t)Cmax, (cuuint64_t)B};
  const cuuint64_t strides[2] = {(cuuint64_t)Hq * 4, (cuuint64_t)Cmax * Hq * 4};
  const cuuint32_t box[3] = {(cuuint32_t)width, (cuuint32_t)R, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(attn), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(GQA_AV_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled (attn) failed (%d)", (int)r);
  return GQA_AV_OK;
}

int current_device(int* dev) {
  cudaError_t e = cudaGetDevice(dev);
  return e == cudaSuccess ? GQA_AV_OK : fail_cuda(e, "cudaGetDevice");
}

// ------------------------------------------------------------ generic path
struct GenPlan {
  int mode, heads, hgroups, tiles, cw, row_par, rows_per_split, nsplit;
  size_t ws_bytes;  // partials only
};

// Whether a tuning asks for anything (the generic kernel takes none).
bool tuning_set(const gqa_av_tuning* t) {
  return t && (t->nsplit || t->dtile || t->rows_per_stage || t->stages || t->early_stages ||
               t->engine || t->split_mode);
}

int make_gen_plan(int dev, int B, int Cmax, int Hq, int Hkv, int D, int mode, GenPlan* p) {
  DeviceInfo di;
  int rc = device_info(dev, &di);
  if (rc) return rc;
  const int G = Hq / Hkv;
  p->mode = mode == GQA_AV_MODE_AUTO ? (G > 1 ? GQA_AV_MODE_GQA : GQA_AV_MODE_PER_HEAD) : mode;
  p->heads = p->mode == GQA_AV_MODE_GQA ? G : 1;
  p->hgroups = Hq / p->heads;
  p->tiles = p->hgroups * B;
  p->cw = D >= kGenThreads ? kGenThreads : (D + 31) / 32 * 32;
  p->row_par = kGenThreads / p->cw;
  // About eight CTAs per SM over the tiles (each thread has a few loads in
  // flight; the kernel waits on memory latency), at least 32 rows a split.
  long long want = p->tiles < 8 * di.sms ? (8LL * di.sms + p->tiles - 1) / p->tiles : 1;
  want = std::max<long long>(1, std::min<long long>(want, (Cmax + 31) / 32));
  p->rows_per_split = static_cast<int>((Cmax + want - 1) / want);
  p->nsplit = (Cmax + p->rows_per_split - 1) / p->rows_per_split;
  if (static_cast<long long>(p->tiles) * p->nsplit > 0x7fffffffLL)
    return fail(GQA_AV_ERR_UNSUPPORTED, "grid too large");
  p->ws_bytes = p->nsplit > 1
                    ? static_cast<size_t>(p->tiles) * p->nsplit * p->heads * D * sizeof(float)
                    : 0;
  return GQA_AV_OK;
}

int run_generic(const float* attn, const void* v, const int32_t* seq_lens, float* out, int B,
                int Cmax, int Hq, int Hkv, int D, int v_dtype, int mode, cudaStream_t stream) {
  if ((reinterpret_cast<uintptr_t>(attn) | reinterpret_cast<uintptr_t>(out)) & 3)
    return fail(GQA_AV_ERR_INVALID, "attn and out must be 4-byte aligned (float)");
  if (reinterpret_cast<uintptr_t>(v) & 1)
    return fail(GQA_AV_ERR_INVALID, "v_cache must be 2-byte aligned (bf16 / fp16)");
  int dev, rc;
  if ((rc = current_device(&dev))) return rc;
  GenPlan gp;
  if ((rc = make_gen_plan(dev, B, Cmax, Hq, Hkv, D, mode, &gp))) return rc;
  Workspace ws;
  if ((rc = workspace(dev, kHeaderBytes + gp.ws_bytes, stream, &ws))) return rc;
  GenericParams p;
  p.attn = attn;
  p.v = static_cast<const uint16_t*>(v);
  p.seq_lens = seq_lens;
  p.out = out;
  p.ws = reinterpret_cast<float*>(static_cast<char*>(ws.base) + kHeaderBytes);
  p.B = B; p.Cmax = Cmax; p.Hq = Hq; p.Hkv = Hkv; p.D = D; p.G = Hq / Hkv;
  p.heads = gp.heads; p.hgroups = gp.hgroups; p.cw = gp.cw; p.row_par = gp.row_par;
  p.rows_per_split = gp.rows_per_split; p.nsplit = gp.nsplit;
  const dim3 grid(static_cast<unsigned>(gp.tiles * gp.nsplit));
  if (v_dtype == GQA_AV_BF16)
    gqa_av_generic_kernel<Bf16Tag><<<grid, kGenThreads, 0, stream>>>(p);
  else
    gqa_av_generic_kernel<Fp16Tag><<<grid, kGenThreads, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail_cuda(e, "generic kernel launch");
  if (gp.nsplit > 1) {
    const int chunks = (gp.heads * D + kGenCombineOut - 1) / kGenCombineOut;
    gqa_av_generic_combine<<<gp.tiles * chunks, kGenThreads, 0, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return fail_cuda(e, "generic combine launch");
  }
  return GQA_AV_OK;
}

int run(const float* attn, const void* v, const int32_t* seq_lens, float* out, int B, int Cmax,
        int Hq, int Hkv, int D, int v_dtype, int mode, const gqa_av_tuning* tuning,
        cudaStream_t stream, const int32_t* block_table = nullptr, int block_size = 0,
        int num_blocks = 0, int max_blocks = 0) {
  g_last_error.clear();
  int rc = check_shape_any_d(B, Cmax, Hq, Hkv, D, v_dtype, mode);
  if (rc) return rc;
  // Contiguous calls that the TMA kernels cannot take (D % 8 != 0, or attn,
  // V or out not 16-byte aligned) run the generic kernel.
  if (!block_table && attn && v && out &&
      (D % 8 != 0 || ((reinterpret_cast<uintptr_t>(attn) | reinterpret_cast<uintptr_t>(v) |
                       reinterpret_cast<uintptr_t>(out)) & 15))) {
    if (tuning_set(tuning))
      return fail(GQA_AV_ERR_UNSUPPORTED,
                  "launch-shape tunings apply to the TMA kernels, which need D %% 8 == 0 and "
                  "16-byte aligned attn, v_cache and out");
    if (reinterpret_cast<uintptr_t>(seq_lens) & 3)
      return fail(GQA_AV_ERR_INVALID, "seq_lens must be 4-byte aligned");
    return run_generic(attn, v, seq_lens, out, B, Cmax, Hq, Hkv, D, v_dtype, mode, stream);
  }
  if ((rc = check_shape(B, Cmax, Hq, Hkv, D, v_dtype, mode))) return rc;
  if (block_table) {
    if (block_size <= 0 || block_size % 8 || num_blocks <= 0 || max_blocks <= 0)
      return fail(GQA_AV_ERR_INVALID,
                  "paged V: block_size=%d must be a positive multiple of 8, num_blocks=%d and "
                  "max_blocks=%d positive", block_size, num_blocks, max_blocks);
    if (static_cast<long long>(max_blocks) * block_size < Cmax)
      return fail(GQA_AV_ERR_INVALID, "paged V: max_blocks x block_size = %lld < Cmax = %d",
                  static_cast<long long>(max_blocks) * block_size, Cmax);
    if (reinterpret_cast<uintptr_t>(block_table) & 3)
      return fail(GQA_AV_ERR_INVALID, "block_table must be 4-byte aligned");
  }
  if (!attn || !v || !out) return fail(GQA_AV_ERR_INVALID, "attn, v_cache and out must be non-NULL");
  if ((reinterpret_cast<uintptr_t>(attn) | reinterpret_cast<uintptr_t>(v) |
       reinterpret_cast<uintptr_t>(out)) & 15)
    return fail(GQA_AV_ERR_UNSUPPORTED, "attn, v_cache and out must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(seq_lens) & 3)
    return fail(GQA_AV_ERR_INVALID, "seq_lens must be 4-byte aligned");
  int dev;
  if ((rc = current_device(&dev))) return rc;
  Plan pl;
  if ((rc = make_plan(dev, B, Cmax, Hq, Hkv, D, v_dtype, mode, tuning, &pl, block_table ? block_size : 0)))
    return rc;
  Workspace ws;
  if ((rc = workspace(dev, kHeaderBytes + pl.ws_bytes, stream, &ws))) return rc;

  Params p;
  memset(&p, 0, sizeof p);
  if (block_table)
    rc = encode_v_map(&p.v_map, v, num_blocks, block_size, Hkv, D, pl.dt, pl.chunk_rows,
                      pl.engine == kEngineTensor);
  else
    rc = encode_v_map(&p.v_map, v, B, Cmax, Hkv, D, pl.dt, pl.R, pl.engine == kEngineTensor);
  if (rc) return rc;
  char* wsb = static_cast<char*>(ws.base);
  fill_params(&p, pl, attn, seq_lens, out, wsb, wsb + kHeaderBytes, B, Cmax, Hq, Hkv, D);
  p.block_table = block_table;
  p.block_size = block_size;
  p.max_blocks = max_blocks;
  p.num_blocks = num_blocks;
  if (p.attn_tma && (rc = encode_attn_map(&p.a_map, attn, B, Cmax, Hq, pl.ap, pl.R))) return rc;

  Kernel kern;
  if (!pick_kernel(v_dtype, kernel_engine(pl), kernel_sel(pl), &kern)) return fail(GQA_AV_ERR_UNSUPPORTED, "no kernel");
  cudaError_t e = launch_call(kern, pl, p, stream);
  if (e != cudaSuccess) return fail_cuda(e, "kernel launch");
  return GQA_AV_OK;
}

}  // namespace

// Programmatic dependent launch, like the main kernel: the combine starts its
// prologue while the main kernel drains and reads the partials only after
// griddepcontrol.wait.
cudaError_t launch_combine(const CombineParams& p, int grid, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kCombineThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e =
      p.balanced == kCombineStream
          ? cudaLaunchKernelEx(&cfg, gqa_av_combine_kernel<kCombineStream>, p)
          : (p.balanced == kCombineBalanced
                 ? cudaLaunchKernelEx(&cfg, gqa_av_combine_kernel<kCombineBalanced>, p)
                 : cudaLaunchKernelEx(&cfg, gqa_av_combine_kernel<kCombineFixed>, p));
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace gqa_av

using namespace gqa_av;

extern "C" {

int gqa_av_decode(const float* attn, const void* v_cache, const int32_t* seq_lens, float* out,
                  int B, int Cmax, int Hq, int Hkv, int D, int v_dtype, int mode, void* stream) {
  return run(attn, v_cache, seq_lens, out, B, Cmax, Hq, Hkv, D, v_dtype, mode, nullptr,
             static_cast<cudaStream_t>(stream));
}

int gqa_av_decode_per_head(const float* attn, const void* v_cache, const int32_t* seq_lens,
                           float* out, int B, int Cmax, int Hq, int Hkv, int D, int v_dtype,
                           void* stream) {
  return run(attn, v_cache, seq_lens, out, B, Cmax, Hq, Hkv, D, v_dtype, GQA_AV_MODE_PER_HEAD,
             nullptr, static_cast<cudaStream_t>(stream));
}

int gqa_av_decode_tuned(const float* attn, const void* v_cache, const int32_t* seq_lens,
                        float* out, int B, int Cmax, int Hq, int Hkv, int D, int v_dtype, int mode,
                        const gqa_av_tuning* tuning, void* stream) {
  return run(attn, v_cache, seq_lens, out, B, Cmax, Hq, Hkv, D, v_dtype, mode, tuning,
             static_cast<cudaStream_t>(stream));
}

int gqa_av_decode_paged(const float* attn, const void* v_pool, const int32_t* block_table,
                        const int32_t* seq_lens, float* out, int B, int Cmax, int Hq, int Hkv,
                        int D, int v_dtype, int block_size, int num_blocks, int max_blocks,
                        int mode, const gqa_av_tuning* tuning, void* stream) {
  if (!block_table) {
    g_last_error.clear();
    return fail(GQA_AV_ERR_INVALID, "block_table must be non-NULL");
  }
  return run(attn, v_pool, seq_lens, out, B, Cmax, Hq, Hkv, D, v_dtype, mode, tuning,
             static_cast<cudaStream_t>(stream), block_table, block_size, num_blocks, max_blocks);
}

int gqa_av_plan(int B, int Cmax, int Hq, int Hkv, int D, int v_dtype, int mode,
                const gqa_av_tuning* tuning, gqa_av_plan_info* info) {
  g_last_error.clear();
  if (!info) return fail(GQA_AV_ERR_INVALID, "info must be non-NULL");
  int dev, rc;
  if ((rc = check_shape_any_d(B, Cmax, Hq, Hkv, D, v_dtype, mode))) return rc;
  if ((rc = current_device(&dev))) return rc;
  if (D % 8 != 0 && !tuning_set(tuning)) {
    // The generic kernel (the plan cannot see pointers: misaligned ones also
    // take it, with this launch).
    GenPlan g;
    if ((rc = make_gen_plan(dev, B, Cmax, Hq, Hkv, D, mode, &g))) return rc;
    memset(info, 0, sizeof *info);
    info->mode = g.mode;
    info->heads_per_cta = g.heads;
    info->head_chunk = std::min(g.heads, kGenHeads);
    info->dtile = g.cw;
    info->rows_per_stage = g.row_par;
    info->nsplit = g.nsplit;
    info->combine_ctas =
        g.nsplit > 1 ? g.tiles * ((g.heads * D + kGenCombineOut - 1) / kGenCombineOut) : 0;
    info->rows_per_split = g.rows_per_split;
    info->tiles = g.tiles;
    info->ctas = g.tiles * g.nsplit;
    info->threads_per_cta = kGenThreads;
    info->engine = kEngineGeneric;
    info->split_mode = 1;
    info->smem_bytes = kGenHeads * kGenThreads * 4;
    info->workspace_bytes = kHeaderBytes + g.ws_bytes;
    return GQA_AV_OK;
  }
  Plan p;
  if ((rc = make_plan(dev, B, Cmax, Hq, Hkv, D, v_dtype, mode, tuning, &p))) return rc;
  info->mode = p.mode;
  info->heads_per_cta = p.heads;
  info->head_chunk = p.gc;
  info->dtile = p.dt;
  info->rows_per_stage = p.R;
  info->stages = p.stages;
  info->early_stages = p.early;
  info->nsplit = p.nsplit;
  info->combine_ctas = p.combine ? p.tiles * p.ctas_per_tile : 0;
  info->rows_per_split = p.rows_per_split;
  info->tiles = p.tiles;
  info->ctas = p.grid;
  info->threads_per_cta = p.engine == kEngineTensor ? mma_threads(p.cvt_warps) : cta_threads(p.gc);
  info->engine = p.engine;
  info->split_mode = p.stream ? 3 : (p.balanced ? 2 : 1);
  info->smem_bytes = p.smem;
  info->ctas_per_sm = p.occ;
  info->workspace_bytes = kHeaderBytes + p.ws_bytes;
  return GQA_AV_OK;
}

size_t gqa_av_workspace_bytes(int B, int Cmax, int Hq, int Hkv, int D, int v_dtype, int mode) {
  gqa_av_plan_info info;
  if (gqa_av_plan(B, Cmax, Hq, Hkv, D, v_dtype, mode, nullptr, &info) != GQA_AV_OK) return 0;
  return info.workspace_bytes;
}

int gqa_av_set_workspace(void* ptr, size_t bytes) {
  g_last_error.clear();
  int dev, rc;
  if ((rc = current_device(&dev))) return rc;
  if (ptr && bytes < kHeaderBytes)
    return fail(GQA_AV_ERR_INVALID, "workspace must hold at least %zu B", kHeaderBytes);
  if (ptr && (reinterpret_cast<uintptr_t>(ptr) & 255))
    return fail(GQA_AV_ERR_INVALID, "workspace must be 256-byte aligned");
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return fail_cuda(e, "cudaDeviceSynchronize");
  std::lock_guard<std::mutex> lk(g_mu);
  Workspace& w = g_ws[dev];
  if (w.base && !w.user) cudaFree(w.base);
  w = Workspace();
  if (ptr) {
    e = cudaMemset(ptr, 0, kHeaderBytes);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail_cuda(e, "zeroing the workspace header");
    w.base = ptr;
    w.bytes = bytes;
    w.user = true;
  }
  return GQA_AV_OK;
}

int gqa_av_device_status(void* stream, int clear) {
  g_last_error.clear();
  int dev, rc;
  if ((rc = current_device(&dev))) return rc;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, "cudaStreamSynchronize");
  // The workspace's word and, once the no-allocation call has run on this
  // device, the word in its fixed array.
  void* words[2] = {nullptr, nullptr};
  {
    std::lock_guard<std::mutex> lk(g_mu);
    words[0] = g_ws[dev].base;
    auto it = g_noalloc_status.find(dev);
    if (it != g_noalloc_status.end()) words[1] = it->second;
  }
  unsigned any = 0;
  for (void* w : words) {
    if (!w) continue;
    unsigned word = 0;
    e = cudaMemcpy(&word, w, sizeof word, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail_cuda(e, "reading the device status word");
    if (clear && word) {
      e = cudaMemset(w, 0, sizeof word);
      if (e == cudaSuccess) e = cudaDeviceSynchronize();
      if (e != cudaSuccess) return fail_cuda(e, "clearing the device status word");
    }
    any |= word;
  }
  if (any)
    return fail(GQA_AV_ERR_DEVICE_TIMEOUT, "a bounded wait ran out on the device (status 0x%x)", any);
  return GQA_AV_OK;
}

const char* gqa_av_status_string(int status) {
  switch (status) {
    case GQA_AV_OK: return "GQA_AV_OK";
    case GQA_AV_ERR_INVALID: return "GQA_AV_ERR_INVALID";
    case GQA_AV_ERR_UNSUPPORTED: return "GQA_AV_ERR_UNSUPPORTED";
    case GQA_AV_ERR_CUDA: return "GQA_AV_ERR_CUDA";
    case GQA_AV_ERR_NOMEM: return "GQA_AV_ERR_NOMEM";
    case GQA_AV_ERR_DEVICE_TIMEOUT: return "GQA_AV_ERR_DEVICE_TIMEOUT";
    default: return "GQA_AV_ERR_UNKNOWN";
  }
}

const char* gqa_av_last_error(void) { return g_last_error.c_str(); }

int gqa_av_version(void) { return 1; }

}  // extern "C"

// ---------------------------------------------------------------------------
// Support for the no-allocation entry point (gqa_av_noalloc.cu). These two
// functions are used only by that entry point and leave the paths above as
// they are.
// ---------------------------------------------------------------------------
namespace gqa_av {

int record_error(int status, const char* msg) { return fail(status, "%s", msg); }

void register_noalloc_status(int dev, void* status_word) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_noalloc_status[dev] = status_word;
}

// One call of the reduction in the default launch shape, with the status
// word and split partials placed in caller-given device scratch laid out as
// [status_bytes][partials]. Leaves the status word as it is (only
// gqa_av_device_status clears it); allocates nothing.
int run_in_scratch(const float* attn, const void* v, const int32_t* seq_lens, float* out, int B,
                   int Cmax, int Hq, int Hkv, int D, int v_dtype, int mode, cudaStream_t stream,
                   void* scratch, size_t status_bytes, size_t scratch_bytes) {
  g_last_error.clear();
  int rc = check_shape(B, Cmax, Hq, Hkv, D, v_dtype, mode);
  if (rc) return rc;
  if (!attn || !v || !out) return fail(GQA_AV_ERR_INVALID, "attn, v_cache and out must be non-NULL");
  if ((reinterpret_cast<uintptr_t>(attn) | reinterpret_cast<uintptr_t>(v) |
       reinterpret_cast<uintptr_t>(out)) & 15)
    return fail(GQA_AV_ERR_UNSUPPORTED, "attn, v_cache and out must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(seq_lens) & 3)
    return fail(GQA_AV_ERR_INVALID, "seq_lens must be 4-byte aligned");
  int dev;
  if ((rc = current_device(&dev))) return rc;
  Plan pl;
  if ((rc = make_plan(dev, B, Cmax, Hq, Hkv, D, v_dtype, mode, nullptr, &pl))) return rc;
  const size_t partial_cap = scratch_bytes - status_bytes;
  if (pl.ws_bytes > partial_cap)
    return fail(GQA_AV_ERR_UNSUPPORTED,
                "no-allocation call: this shape needs %zu B of split partials, the fixed scratch "
                "holds %zu B (use gqa_av_decode)",
                pl.ws_bytes, partial_cap);
  char* base = static_cast<char*>(scratch);
  cudaError_t e;

  Params p;
  memset(&p, 0, sizeof p);
  if ((rc = encode_v_map(&p.v_map, v, B, Cmax, Hkv, D, pl.dt, pl.R, pl.engine == kEngineTensor))) return rc;
  fill_params(&p, pl, attn, seq_lens, out, base, base + status_bytes, B, Cmax, Hq, Hkv, D);
  if (p.attn_tma && (rc = encode_attn_map(&p.a_map, attn, B, Cmax, Hq, pl.ap, pl.R))) return rc;

  Kernel kern;
  if (!pick_kernel(v_dtype, kernel_engine(pl), kernel_sel(pl), &kern)) return fail(GQA_AV_ERR_UNSUPPORTED, "no kernel");
  e = launch_call(kern, pl, p, stream);
  if (e != cudaSuccess) return fail_cuda(e, "kernel launch");
  return GQA_AV_OK;
}

int noalloc_scratch(int dev, void** ptr, size_t* status_bytes, size_t* bytes);  // gqa_av_noalloc.cu

// Self-test of the failure path: the FMA kernel in its default launch shape
// for this call, with the producer withholding every full split's last stage
// (nothing of it is ever issued, so no copy is in flight when the CTA leaves)
// and the consumers' wait for a stage bounded by `wait_ns`. The consumers'
// wait for the withheld stage runs out: they set the status word (in the
// workspace, or in the no-allocation call's fixed array) and return through
// the same barriers as on any other timeout. `out` is left unspecified.
int selftest_wait_timeout(const float* attn, const void* v, const int32_t* seq_lens, float* out,
                          int B, int Cmax, int Hq, int Hkv, int D, int v_dtype, long long wait_ns,
                          int scratch_kind, cudaStream_t stream) {
  g_last_error.clear();
  int rc = check_shape(B, Cmax, Hq, Hkv, D, v_dtype, GQA_AV_MODE_AUTO);
  if (rc) return rc;
  if (!attn || !v || !out) return fail(GQA_AV_ERR_INVALID, "attn, v_cache and out must be non-NULL");
  if ((reinterpret_cast<uintptr_t>(attn) | reinterpret_cast<uintptr_t>(v) |
       reinterpret_cast<uintptr_t>(out)) & 15)
    return fail(GQA_AV_ERR_UNSUPPORTED, "attn, v_cache and out must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(seq_lens) & 3)
    return fail(GQA_AV_ERR_INVALID, "seq_lens must be 4-byte aligned");
  if (wait_ns < 1000 || wait_ns > kWaitTimeoutNs)
    return fail(GQA_AV_ERR_INVALID, "wait_ns=%lld must be in [1000, %lld]", wait_ns,
                kWaitTimeoutNs);
  if (scratch_kind != 0 && scratch_kind != 1)
    return fail(GQA_AV_ERR_INVALID, "scratch=%d must be 0 (workspace) or 1 (fixed array)",
                scratch_kind);
  int dev;
  if ((rc = current_device(&dev))) return rc;
  gqa_av_tuning t;
  memset(&t, 0, sizeof t);
  t.engine = kEngineFma;
  Plan pl;
  if ((rc = make_plan(dev, B, Cmax, Hq, Hkv, D, v_dtype, GQA_AV_MODE_AUTO, &t, &pl))) return rc;
  // Every full split must have a stage after the one issued before the length
  // is read, or nothing would be withheld.
  if (pl.early != 1 || pl.rows_per_split < 2 * pl.R)
    return fail(GQA_AV_ERR_UNSUPPORTED,
                "self-test needs splits of at least two stages (rows_per_split %d, R %d)",
                pl.rows_per_split, pl.R);
  char* base = nullptr;
  size_t status_bytes = kHeaderBytes;
  if (scratch_kind == 1) {
    void* ptr = nullptr;
    size_t bytes = 0;
    if ((rc = noalloc_scratch(dev, &ptr, &status_bytes, &bytes))) return rc;
    if (pl.ws_bytes > bytes - status_bytes)
      return fail(GQA_AV_ERR_UNSUPPORTED, "self-test shape needs %zu B of split partials",
                  pl.ws_bytes);
    base = static_cast<char*>(ptr);
  } else {
    Workspace ws;
    if ((rc = workspace(dev, kHeaderBytes + pl.ws_bytes, stream, &ws))) return rc;
    base = static_cast<char*>(ws.base);
  }
  Params p;
  memset(&p, 0, sizeof p);
  if ((rc = encode_v_map(&p.v_map, v, B, Cmax, Hkv, D, pl.dt, pl.R, false))) return rc;
  fill_params(&p, pl, attn, seq_lens, out, base, base + status_bytes, B, Cmax, Hq, Hkv, D);
  if (p.attn_tma && (rc = encode_attn_map(&p.a_map, attn, B, Cmax, Hq, pl.ap, pl.R))) return rc;
  p.full_wait_ns = wait_ns;
  p.withhold_last = 1;
  Kernel kern;
  if (!pick_kernel(v_dtype, pl.engine, kernel_sel(pl), &kern))
    return fail(GQA_AV_ERR_UNSUPPORTED, "no kernel");
  cudaError_t e = launch_call(kern, pl, p, stream);
  if (e != cudaSuccess) return fail_cuda(e, "kernel launch");
  return GQA_AV_OK;
}

}  // namespace gqa_av

extern "C" int gqa_av_selftest_wait_timeout(const float* attn, const void* v_cache,
                                            const int32_t* seq_lens, float* out, int B, int Cmax,
                                            int Hq, int Hkv, int D, int v_dtype,
                                            long long wait_ns, int scratch, void* stream) {
  return gqa_av::selftest_wait_timeout(attn, v_cache, seq_lens, out, B, Cmax, Hq, Hkv, D,
                                       v_dtype, wait_ns, scratch,
                                       static_cast<cudaStream_t>(stream));
}
