// GQA AV decode reduction kernel for sm_103a (GB300).
//
// Operation (page "pytorch/executorch pull 21063", summary paragraph):
//   out[b, q_h, d] = sum_{c < L_b} attn[b, c, q_h] * V[b, c, q_h / G, d].
//
// One CTA owns a tile (head group, b, d-tile) and one context split of it.
// In GQA-reuse mode a head group is the G query heads of one KV head, so each
// V row is fetched from HBM once and used for all G heads (the GQA-reuse
// paragraph on the same page); in per-head mode a head group is one query
// head and V rows are fetched once per query head.
//
// Warp roles:
//   * warp kConsumerWarps (the producer): lane 0 streams V rows with 4-D TMA
//     tensor loads into a multi-stage shared-memory ring; all 32 lanes copy the
//     matching attn weights with cp.async. Both signal one "full" mbarrier per
//     stage.
//   * warps 0..kConsumerWarps-1 (consumers): thread t owns 8 adjacent output
//     columns of one head chunk and a row slot; for every V row of its slot it
//     widens 8 bf16/fp16 values to fp32 and does GC x 8 FMAs into registers,
//     then releases the stage through an "empty" mbarrier.
// After the context loop the row slots are summed in shared memory in a fixed
// order. A split that is alone writes `out` directly; otherwise it writes its
// partial to the workspace and takes a ticket; the last CTA of the tile sums
// all partials in split order and writes `out`, so results are bitwise
// reproducible and independent of CTA arrival order. Every mbarrier wait is
// bounded by a %globaltimer deadline; on expiry the CTA sets the device status
// word, lets its own copies in flight land, and returns.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gqa_av {

constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kThreads = kConsumerThreads + 32;
constexpr int kMaxStages = 8;

// Device status word bits.
constexpr unsigned kErrFullWait = 1u;
constexpr unsigned kErrEmptyWait = 2u;
constexpr unsigned kErrDrain = 4u;

struct alignas(64) Params {
  CUtensorMap v_map;            // V as 4-D {D, Hkv, Cmax, B}; box {dt, 1, R, 1}
  const float* attn;            // [B, Cmax, Hq]
  const int32_t* seq_lens;      // [B] or null
  float* out;                   // [B, Hq, D]
  float* ws;                    // [tiles][nsplit][heads * dt] partials
  unsigned int* tickets;        // [tiles], zero between calls
  unsigned int* status;         // device status word
  int B, Cmax, Hq, Hkv, D, G;
  int heads;                    // query heads per CTA
  int hgroups;                  // Hq / heads
  int dt;                       // output columns per CTA
  int ndt;                      // D / dt
  int ct;                       // dt / 8 column threads
  int nc;                       // heads / GC head chunks
  int row_par;                  // consumer row slots
  int R;                        // rows per stage
  int stages;
  int rows_per_split;
  int nsplit;
  int ap;                       // floats per attn row in shared memory
  int avec;                     // floats per attn cp.async (1, 2 or 4)
  uint32_t v_stage_bytes;       // R * dt * 2
  uint32_t a_off;               // shared-memory offset of the attn ring
  uint32_t bar_off;             // shared-memory offset of the mbarriers
  long long timeout_ns;         // bound on every mbarrier wait
};

// ---------------------------------------------------------------------------
// PTX helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase of `parity` to complete; false if `timeout_ns` passed.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, long long timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (static_cast<long long>(global_timer_ns() - t0) > timeout_ns) return false;
  }
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// 4-D tiled TMA load global -> shared, completion counted on `bar` in bytes.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int x0, int x1,
                                            int x2, int x3, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cta.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x0), "r"(x1), "r"(x2), "r"(x3), "r"(bar),
      "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

template <int BYTES>
__device__ __forceinline__ void cp_async(uint32_t dst, const void* src) {
  if constexpr (BYTES == 16) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
  } else {
    asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" ::"r"(dst), "l"(src), "n"(BYTES)
                 : "memory");
  }
}

// Arrive on `bar` once every cp.async this thread issued so far has landed.
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory");
}

// ---------------------------------------------------------------------------
// Element widening: 8 packed 16-bit values -> 8 fp32 (exact for bf16/fp16).
// ---------------------------------------------------------------------------
struct Bf16Tag {};
struct Fp16Tag {};

__device__ __forceinline__ void widen8(Bf16Tag, const uint4 raw, float (&v)[8]) {
  // bfloat16 is the upper half of a binary32 pattern.
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ void widen8(Fp16Tag, const uint4 raw, float (&v)[8]) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
    float2 f = __half22float2(h);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}

template <int GC>
__device__ __forceinline__ void load_weights(const float* a, float (&w)[GC]) {
  if constexpr (GC % 4 == 0) {
#pragma unroll
    for (int g = 0; g < GC; g += 4) {
      const float4 x = *reinterpret_cast<const float4*>(a + g);
      w[g] = x.x; w[g + 1] = x.y; w[g + 2] = x.z; w[g + 3] = x.w;
    }
  } else if constexpr (GC % 2 == 0) {
#pragma unroll
    for (int g = 0; g < GC; g += 2) {
      const float2 x = *reinterpret_cast<const float2*>(a + g);
      w[g] = x.x; w[g + 1] = x.y;
    }
  } else {
#pragma unroll
    for (int g = 0; g < GC; ++g) w[g] = a[g];
  }
}

// ---------------------------------------------------------------------------
// The kernel. Tag selects the V element type, GC the heads per thread.
// ---------------------------------------------------------------------------
template <typename Tag, int GC>
__global__ void __launch_bounds__(kThreads, (GC <= 8 ? 2 : 1))
gqa_av_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) uint8_t smem[];

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  // Tile and split of this CTA; head group is the slowest index.
  const int tiles_per_hg = p.B * p.ndt;
  const int tile = blockIdx.x / p.nsplit;
  const int split = blockIdx.x - tile * p.nsplit;
  const int hg = tile / tiles_per_hg;
  const int rem = tile - hg * tiles_per_hg;
  const int b = rem / p.ndt;
  const int dti = rem - b * p.ndt;
  const int h0 = hg * p.heads;            // first query head of the CTA
  const int kv_h = h0 / p.G;              // its KV head (all heads of the CTA share it)
  const int d0 = dti * p.dt;

  int L = p.seq_lens ? p.seq_lens[b] : p.Cmax;
  L = L < 0 ? 0 : (L > p.Cmax ? p.Cmax : L);
  const int nsplit_b = L > 0 ? (L + p.rows_per_split - 1) / p.rows_per_split : 1;
  if (split >= nsplit_b) return;          // whole CTA: no context left for it
  const int c_begin = split * p.rows_per_split;
  const int c_end = min(c_begin + p.rows_per_split, L);
  const int n_iters = c_end > c_begin ? (c_end - c_begin + p.R - 1) / p.R : 0;
  const int tile_elems = p.heads * p.dt;

  uint8_t* vring = smem;
  float* aring = reinterpret_cast<float*>(smem + p.a_off);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.bar_off);
  volatile int& s_flag = *reinterpret_cast<int*>(bars + 2 * kMaxStages);
  const uint32_t full0 = smem_addr(bars);
  const uint32_t empty0 = smem_addr(bars + kMaxStages);

  if (tid == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(full0 + 8 * s, 1 + 32);           // expect_tx arrival + 32 cp.async arrivals
      mbar_init(empty0 + 8 * s, kConsumerWarps);  // one arrival per consumer warp
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    s_flag = 0;
  }
  __syncthreads();

  // ----------------------------------------------------------------- producer
  if (warp == kConsumerWarps) {
    const uint64_t policy = evict_first_policy();
    const int per_row = p.heads / p.avec;
    int issued = 0;
    bool ok = true;
    for (int it = 0; it < n_iters; ++it) {
      const int stage = it % p.stages;
      const uint32_t parity = ((it / p.stages) & 1) ^ 1;
      if (!mbar_wait(empty0 + 8 * stage, parity, p.timeout_ns)) {
        atomicOr(p.status, kErrEmptyWait);
        ok = false;
        break;
      }
      const int c0 = c_begin + it * p.R;
      const int rows = min(p.R, c_end - c0);
      const uint32_t full = full0 + 8 * stage;
      if (lane == 0) {
        mbar_arrive_expect_tx(full, p.v_stage_bytes);
        tma_load_4d(smem_addr(vring + (size_t)stage * p.v_stage_bytes), &p.v_map, d0, kv_h, c0, b,
                    full, policy);
      }
      const float* src = p.attn + ((size_t)b * p.Cmax + c0) * p.Hq + h0;
      const uint32_t dst = smem_addr(aring + (size_t)stage * p.R * p.ap);
      const int n = rows * per_row;
      if (p.avec == 4) {
        for (int i = lane; i < n; i += 32) {
          const int r = i / per_row, k = i - r * per_row;
          cp_async<16>(dst + 4u * (r * p.ap + 4 * k), src + (size_t)r * p.Hq + 4 * k);
        }
      } else if (p.avec == 2) {
        for (int i = lane; i < n; i += 32) {
          const int r = i / per_row, k = i - r * per_row;
          cp_async<8>(dst + 4u * (r * p.ap + 2 * k), src + (size_t)r * p.Hq + 2 * k);
        }
      } else {
        for (int i = lane; i < n; i += 32) {
          const int r = i / per_row, k = i - r * per_row;
          cp_async<4>(dst + 4u * (r * p.ap + k), src + (size_t)r * p.Hq + k);
        }
      }
      cp_async_arrive_noinc(full);
      issued = it + 1;
    }
    cp_async_wait_all();
    if (!ok) {
      // Let every TMA load this CTA issued land before the CTA can exit.
      for (int it = 0; it < issued; ++it) {
        const int stage = it % p.stages;
        // Only the latest use of each stage can still be in flight.
        if (it + p.stages < issued) continue;
        if (!mbar_wait(full0 + 8 * stage, (it / p.stages) & 1, p.timeout_ns))
          atomicOr(p.status, kErrDrain);
      }
    }
    return;
  }

  // ---------------------------------------------------------------- consumers
  const int slots = p.ct * p.nc;
  const int my_col = tid % p.ct;
  const int my_chunk = (tid / p.ct) % p.nc;
  const int my_slot = tid / slots;
  const bool active = my_slot < p.row_par;

  float acc[GC][8];
#pragma unroll
  for (int g = 0; g < GC; ++g)
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[g][k] = 0.f;

  bool ok = true;
  for (int it = 0; it < n_iters; ++it) {
    const int stage = it % p.stages;
    if (!mbar_wait(full0 + 8 * stage, (it / p.stages) & 1, p.timeout_ns)) {
      atomicOr(p.status, kErrFullWait);
      ok = false;
      break;
    }
    const int rows = min(p.R, c_end - (c_begin + it * p.R));
    const uint16_t* vst =
        reinterpret_cast<const uint16_t*>(vring + (size_t)stage * p.v_stage_bytes) + my_col * 8;
    const float* ast = aring + (size_t)stage * p.R * p.ap + my_chunk * GC;
    if (active) {
#pragma unroll 2
      for (int r = my_slot; r < rows; r += p.row_par) {
        const uint4 raw = *reinterpret_cast<const uint4*>(vst + (size_t)r * p.dt);
        float v[8];
        widen8(Tag{}, raw, v);
        float w[GC];
        load_weights<GC>(ast + (size_t)r * p.ap, w);
#pragma unroll
        for (int g = 0; g < GC; ++g)
#pragma unroll
          for (int k = 0; k < 8; ++k) acc[g][k] = fmaf(w[g], v[k], acc[g][k]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * stage);
  }
  if (!ok) s_flag = 1;
  consumer_sync();
  if (s_flag) return;  // the producer drains in-flight copies before exiting

  // Row slots -> one partial per (head, column), summed in slot order.
  float* red = reinterpret_cast<float*>(smem);  // the V ring is free now
  if (active) {
    float* dst = red + (size_t)my_slot * tile_elems + (size_t)(my_chunk * GC) * p.dt + my_col * 8;
#pragma unroll
    for (int g = 0; g < GC; ++g) {
      float4* q = reinterpret_cast<float4*>(dst + (size_t)g * p.dt);
      q[0] = make_float4(acc[g][0], acc[g][1], acc[g][2], acc[g][3]);
      q[1] = make_float4(acc[g][4], acc[g][5], acc[g][6], acc[g][7]);
    }
  }
  consumer_sync();

  const bool alone = nsplit_b == 1;
  float* part = p.ws + ((size_t)tile * p.nsplit + split) * tile_elems;
  for (int e = tid * 4; e < tile_elems; e += kConsumerThreads * 4) {
    float4 s = *reinterpret_cast<const float4*>(red + e);
    for (int r = 1; r < p.row_par; ++r) {
      const float4 x = *reinterpret_cast<const float4*>(red + (size_t)r * tile_elems + e);
      s.x += x.x; s.y += x.y; s.z += x.z; s.w += x.w;
    }
    if (alone) {
      const int h = e / p.dt, dd = e - h * p.dt;
      *reinterpret_cast<float4*>(p.out + ((size_t)b * p.Hq + h0 + h) * p.D + d0 + dd) = s;
    } else {
      __stcg(reinterpret_cast<float4*>(part + e), s);
    }
  }
  if (alone) return;

  // Deterministic split combine: the last CTA of the tile sums in split order.
  __threadfence();
  consumer_sync();
  if (tid == 0) {
    const unsigned prev = atomicAdd(p.tickets + tile, 1u);
    s_flag = (prev == static_cast<unsigned>(nsplit_b - 1)) ? 2 : 0;
  }
  consumer_sync();
  if (s_flag != 2) return;
  __threadfence();
  const float* base = p.ws + (size_t)tile * p.nsplit * tile_elems;
  for (int e = tid * 4; e < tile_elems; e += kConsumerThreads * 4) {
    float4 s = __ldcg(reinterpret_cast<const float4*>(base + e));
    for (int r = 1; r < nsplit_b; ++r) {
      const float4 x = __ldcg(reinterpret_cast<const float4*>(base + (size_t)r * tile_elems + e));
      s.x += x.x; s.y += x.y; s.z += x.z; s.w += x.w;
    }
    const int h = e / p.dt, dd = e - h * p.dt;
    *reinterpret_cast<float4*>(p.out + ((size_t)b * p.Hq + h0 + h) * p.D + d0 + dd) = s;
  }
  if (tid == 0) p.tickets[tile] = 0u;
}

// Launch entry for one (element type, head chunk) instantiation.
template <typename Tag, int GC>
cudaError_t launch(const Params& p, int grid, int smem_bytes, cudaStream_t stream);

template <typename Tag, int GC>
cudaError_t occupancy(int smem_limit, int smem_bytes, int* ctas_per_sm);

}  // namespace gqa_av
