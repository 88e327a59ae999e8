// GQA AV decode reduction kernels for sm_103a (GB300).
//
// Operation (page "pytorch/executorch pull 21063", summary paragraph):
//   out[b, q_h, d] = sum_{c < L_b} attn[b, c, q_h] * V[b, c, q_h / G, d].
//
// gqa_av_kernel: one CTA owns a tile (head group, b, d-tile) and one context
// split of it. In GQA-reuse mode a head group is the G query heads of one KV
// head, so each V row is fetched from HBM once and used for all G heads (the
// GQA-reuse paragraph on the same page); in per-head mode a head group is one
// query head and V rows are fetched once per query head.
//
// Warp roles:
//   * producer (warp kConsumerWarps): lane 0 streams V rows with 4-D TMA
//     tensor loads into a multi-stage shared-memory ring, and their attn
//     weights with a 3-D TMA box (head groups of a multiple of 4 heads) or,
//     otherwise, by cp.async from all 32 lanes. Both signal one "full"
//     mbarrier per stage; a slot is refilled once every consumer warp has
//     released it ("empty" mbarrier). The first stage(s) are issued before the
//     sequence length is read.
//   * consumers (warps 0..kConsumerWarps-1): thread t owns 8 adjacent output
//     columns of one head chunk and a row slot; for every V row of its slot it
//     widens 8 bf16/fp16 values to fp32 and does GC x 8 FMAs (packed f32x2,
//     each lane rounded like fmaf) into registers.
// After the context loop the row slots are summed through shared memory in
// slot order. A tile whose context fits one split writes `out`; otherwise
// each split writes its partial to the workspace and gqa_av_combine_kernel,
// launched next on the same stream, sums the partials of every (tile, column)
// in split order. Results are bitwise reproducible.
//
// Both kernels use programmatic dependent launch: each starts its prologue
// while the previous kernel in the stream drains, and touches data of earlier
// kernels only after griddepcontrol.wait. Every mbarrier wait is bounded by a
// %globaltimer deadline; on expiry the CTA sets the device status word, lets
// its own copies in flight land, and returns.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gqa_av {

// Consumer warps per CTA. A sub-partition's register file is shared by its
// warps: with the producer warp, 13 warps put 4 on one sub-partition and leave
// 128 registers a thread (enough up to 8 heads a thread; 12 heads need the 168
// that 9 warps leave). Measured on the Llama-size shape: 12 consumer warps
// beat 8, 11 and 15.
__host__ __device__ constexpr int consumer_warps(int gc) { return gc >= 12 ? 8 : 12; }
__host__ __device__ constexpr int cta_threads(int gc) { return 32 * (consumer_warps(gc) + 1); }
constexpr int kMaxStages = 8;
constexpr int kCombineThreads = 128;
// Partials a combine thread loads at once.
constexpr int kCombineBatch = 8;

// Device status word bits.
constexpr unsigned kErrFullWait = 1u;
constexpr unsigned kErrEmptyWait = 2u;
constexpr unsigned kErrDrain = 4u;

struct alignas(64) Params {
  CUtensorMap v_map;            // V as 4-D {D, Hkv, Cmax, B}; box {dt, 1, R, 1}
  CUtensorMap a_map;            // attn as 3-D {Hq, Cmax, B}; box {ap, R, 1} (when attn_tma)
  const float* attn;            // [B, Cmax, Hq]
  const int32_t* seq_lens;      // [B] or null
  float* out;                   // [B, Hq, D]
  float* ws;                    // split partials: [tiles][nsplit][heads * dt], or one slot a CTA
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
  int nsplit;                   // context splits per tile
  int ap;                       // floats per attn row in shared memory
  int avec;                     // floats per attn cp.async (1, 2 or 4)
  int attn_tma;                 // attn weights by TMA (Hq % 4 == 0) instead of cp.async
  uint32_t a_stage_bytes;       // R * ap * 4
  uint32_t v_stage_bytes;       // R * dt * 2
  uint32_t a_off;               // shared-memory offset of the attn ring
  uint32_t bar_off;             // shared-memory offset of the mbarriers
  int early_stages;             // stages issued before the sequence length is read (>= 1)
  long long timeout_ns;         // bound on every mbarrier wait but the one below
  long long full_wait_ns;       // FMA kernel: bound on the consumers' waits for a stage
  int withhold_last;            // self-test of the failure path (FMA kernel): the producer
                                // issues no copy for a split's last stage, so the
                                // consumers' wait for it runs out (0 in every normal call)
  // Tensor-core kernel only.
  int v_halves;                 // 64-column V boxes per stage (1 or 2)
  uint32_t b_off;               // shared-memory offset of the B (weights) ring
  uint32_t tmem_cols;           // tensor-memory columns allocated (4 x N, power of 2 >= 32)
  int cvt_warps;                // weight-conversion warps (2 or 4)
  int split_units;              // CTAs the batch's context is spread over (balanced, streamed)
  int balanced;                 // splits balanced over the batch's lengths (else fixed)
  uint32_t lens_off;            // streamed kernel: shared-memory offset of the lengths
  // Paged V: the tensor map is over a pool of blocks {D, Hkv, block_size,
  // num_blocks}; a stage's rows come as chunk_rows-row boxes from the blocks
  // that hold them (block_table[b][c / block_size]). Contiguous V: null table,
  // chunk_rows = R.
  const int32_t* block_table;   // [B, max_blocks] or null
  int block_size, max_blocks, num_blocks;
  int chunk_rows;               // rows per V box
};

// The split combine: out[tile column] = sum over the tile's splits with
// context, ws[tile][s][column], in split order.
struct CombineParams {
  const float* ws;              // [tiles][nsplit][tile_elems], or one slot a CTA (balanced)
  const int32_t* seq_lens;      // [B] or null
  float* out;                   // [B, Hq, D]
  int B, Cmax, Hq, D;
  int heads, dt, ndt;
  int rows_per_split, nsplit;
  int tile_elems;               // heads * dt
  int parts;                    // threads per column (fixed chunks of splits)
  int cols_per_cta;             // float4 columns per CTA (kCombineThreads / parts)
  int ctas_per_tile;
  int balanced;                 // 0 fixed splits, 1 length-balanced, 2 streamed
  int R, hgroups, split_units;  // their stage rows, head groups and CTA count
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

// One potentially blocking test of the phase of `parity`: the thread is
// suspended until the phase completes or about `hint_ns` pass, so a waiting
// warp takes no issue slots from the warps that do the work.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Waits for the phase of `parity` to complete; false if `timeout_ns` passed.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, long long timeout_ns) {
  if (mbar_try_wait(bar, parity, 100000u)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity, 100000u)) return true;
    if (static_cast<long long>(global_timer_ns() - t0) > timeout_ns) return false;
  }
}

// The same test without a suspend hint: the thread polls, so it resumes within
// a few tens of nanoseconds of the phase completing (for waits on the
// critical path of a pipeline).
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
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

// Polling wait for the phase of `parity`; false if `timeout_ns` passed.
__device__ __forceinline__ bool mbar_poll(uint32_t bar, uint32_t parity, long long timeout_ns) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    for (int i = 0; i < 64; ++i)
      if (mbar_test(bar, parity)) return true;
    if (static_cast<long long>(global_timer_ns() - t0) > timeout_ns) return false;
  }
}

// Programmatic dependent launch: wait until the previous kernel in the stream
// has completed and its memory is visible (a no-op without such a launch),
// and allow the next kernel to start its own prologue.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Named barrier `id` of `count` threads (a multiple of 32). The warp is
// reconverged first and the unaligned form is used, so a warp whose lanes
// left divergent code apart still arrives as one warp.
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t count) {
  __syncwarp();
  asm volatile("barrier.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void named_arrive(uint32_t id, uint32_t count) {
  __syncwarp();
  asm volatile("barrier.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
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

// 3-D tiled TMA load global -> shared, completion counted on `bar` in bytes.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x0, int x1,
                                            int x2, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x0), "r"(x1), "r"(x2), "r"(bar), "l"(policy)
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

// Named barrier 1 of the consumer warps only (the producer warp does not
// join). Reconverges the warp first (named_sync): on the path where a bounded
// wait ran out, lanes leave their wait loops at different times.
template <int kConsumerThreads>
__device__ __forceinline__ void consumer_sync() {
  named_sync(1, kConsumerThreads);
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

__device__ __forceinline__ void add4(float4& s, const float4 x) {
  s.x += x.x; s.y += x.y; s.z += x.z; s.w += x.w;
}

// s += src[lo * stride] + ... + src[(hi-1) * stride], added in index order;
// the loads of each batch are issued together. kGlobal reads through L2 only.
template <bool kGlobal>
__device__ __forceinline__ void sum_strided(float4& s, const float4* src, size_t stride, int lo,
                                            int hi) {
  constexpr int kBatch = kCombineBatch;
  for (int i0 = lo; i0 < hi; i0 += kBatch) {
    float4 x[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i)
      if (i0 + i < hi) x[i] = kGlobal ? __ldcg(src + (i0 + i) * stride) : src[(i0 + i) * stride];
#pragma unroll
    for (int i = 0; i < kBatch; ++i)
      if (i0 + i < hi) add4(s, x[i]);
  }
}

// TMA row and outermost coordinates of context row c of sequence b: (c, b)
// for a contiguous cache, (c % block_size, block_table[b][c / block_size])
// for a paged one. Rows at or past Cmax, and block indices outside the pool,
// land outside the tensor map, which the TMA unit fills with zeros.
__device__ __forceinline__ int2 v_row_coord(const Params& p, int b, int c) {
  if (!p.block_table) return make_int2(c, b);
  if (c >= p.Cmax) return make_int2(0, p.num_blocks);
  const int j = c / p.block_size;
  return make_int2(c - j * p.block_size, p.block_table[(size_t)b * p.max_blocks + j]);
}

// ---------------------------------------------------------------------------
// Length-balanced splits (the tensor-core kernel and its combine).
//
// The context rows of the whole batch are spread evenly over `units` CTAs,
// whatever the lengths: sequence b (length L_b, ceil(L_b / R) stages of R
// rows) is cut into n_b = max(1, ceil(ceil(L_b / R) / sps)) splits of sps
// stages, where sps = ceil(K * sum_b ceil(L_b / R) / units) and K = hgroups *
// ndt is the number of tiles of one sequence. CTA u takes tile k = u % K of
// its sequence and batch split q = u / K, which is split q - P_b of the
// sequence b with P_b <= q < P_b + n_b (P_b = n_0 + ... + n_{b-1}); at most
// units + K * B CTAs have work and the rest exit. A split's partial is slot u
// of the workspace, so the partials of one tile lie K slots apart.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int clamped_len(const int32_t* seq_lens, int b, int Cmax) {
  const int L = seq_lens ? seq_lens[b] : Cmax;
  return L < 0 ? 0 : (L > Cmax ? Cmax : L);
}

// The same through the read-only data path: the lengths are read by every CTA
// of a call, so CTAs on one SM share them in L1 instead of queueing on one L2
// line. Only for reads after the grid-dependency wait (nothing of them can be
// cached from before it) of lengths no kernel writes while this one runs.
__device__ __forceinline__ int clamped_len_ro(const int32_t* seq_lens, int b, int Cmax) {
  const int L = seq_lens ? __ldg(seq_lens + b) : Cmax;
  return L < 0 ? 0 : (L > Cmax ? Cmax : L);
}

__device__ __forceinline__ int balanced_splits_of(int L, int R, int sps) {
  const int n = ((L + R - 1) / R + sps - 1) / sps;
  return n > 1 ? n : 1;
}

// Stages per split. Warp-collective: all 32 lanes take part.
__device__ __forceinline__ int balanced_sps(const int32_t* seq_lens, int B, int Cmax, int R, int K,
                                            int units) {
  long long s = 0;
  for (int b = threadIdx.x & 31; b < B; b += 32)
    s += (clamped_len(seq_lens, b, Cmax) + R - 1) / R;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  const long long sps = (s * K + units - 1) / units;
  return sps > 1 ? static_cast<int>(sps) : 1;
}

struct BalancedSplit {
  int b, L;        // sequence and its clamped length
  int split, n;    // split of the sequence and the sequence's split count
  int found;       // 0: the batch has fewer splits than q + 1
};

// Sequence and split of batch split q. Warp-collective.
__device__ __forceinline__ BalancedSplit balanced_find(const int32_t* seq_lens, int B, int Cmax,
                                                       int R, int sps, int q) {
  const int lane = threadIdx.x & 31;
  int base = 0;  // splits of the sequences before this chunk of 32
  for (int b0 = 0; b0 < B; b0 += 32) {
    const int b = b0 + lane;
    const int L = b < B ? clamped_len(seq_lens, b, Cmax) : 0;
    const int n = b < B ? balanced_splits_of(L, R, sps) : 0;
    int incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, n > 0 && q >= base + incl - n && q < base + incl);
    if (hit) {
      const int src = __ffs(hit) - 1;
      BalancedSplit r;
      r.b = b0 + src;
      r.L = __shfl_sync(0xffffffffu, L, src);
      r.n = __shfl_sync(0xffffffffu, n, src);
      r.split = q - base - __shfl_sync(0xffffffffu, incl - n, src);
      r.found = 1;
      return r;
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
  BalancedSplit none{0, 0, 0, 0, 0};
  return none;
}

// P_b (splits of the sequences before b) and n_b. Warp-collective.
__device__ __forceinline__ int2 balanced_prefix(const int32_t* seq_lens, int Cmax, int R, int sps,
                                                int b) {
  int s = 0;
  for (int i = threadIdx.x & 31; i < b; i += 32)
    s += balanced_splits_of(clamped_len(seq_lens, i, Cmax), R, sps);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return make_int2(s, balanced_splits_of(clamped_len(seq_lens, b, Cmax), R, sps));
}

// ---------------------------------------------------------------------------
// Streamed schedule (the streamed tensor-core kernel, gqa_av_stream.cuh, and
// its combine): sequence b has stream_stages(L_b, R) stages in each of its K
// tiles; tile column k lists them sequence after sequence, T = sum_b of them;
// group g of Ug takes stages [stream_first(T, g, Ug), stream_first(T, g + 1,
// Ug)) of every column (CTA u = g * K + k takes column k).
// ---------------------------------------------------------------------------
__device__ __forceinline__ int stream_stages(int L, int R) {
  const int n = (L + R - 1) / R;
  return n > 1 ? n : 1;
}

__device__ __forceinline__ long long stream_first(long long T, int g, int Ug) {
  return T * g / Ug;
}

// The group whose range holds stage x: the largest g with stream_first(T, g, Ug) <= x.
__device__ __forceinline__ int stream_owner(long long T, long long x, int Ug) {
  return static_cast<int>(((x + 1) * Ug - 1) / T);
}

// Stages a column holds in all (x) and before sequence b (y). Warp-collective.
__device__ __forceinline__ longlong2 stream_prefix(const int32_t* seq_lens, int B, int Cmax, int R,
                                                   int b) {
  long long tot = 0, pre = 0;
  for (int i = threadIdx.x & 31; i < B; i += 32) {
    const int n = stream_stages(clamped_len(seq_lens, i, Cmax), R);
    tot += n;
    if (i < b) pre += n;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    tot += __shfl_xor_sync(0xffffffffu, tot, o);
    pre += __shfl_xor_sync(0xffffffffu, pre, o);
  }
  return make_longlong2(tot, pre);
}

// Two fp32 lanes in one 64-bit register pair, and the packed FMA on them:
// acc.lo += w * v.lo, acc.hi += w * v.hi, each rounded like fmaf.
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack2(uint64_t x, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(x));
}
__device__ __forceinline__ void ffma2(uint64_t& acc, uint64_t w2, uint64_t v2) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(w2), "l"(v2));
}

// ---------------------------------------------------------------------------
// The main kernel. Tag selects the V element type, GC the heads per thread.
// ---------------------------------------------------------------------------
template <typename Tag, int GC>
__global__ void __launch_bounds__(cta_threads(GC), 1)
gqa_av_kernel(const __grid_constant__ Params p) {
  constexpr int kConsumerWarps = consumer_warps(GC);
  constexpr int kConsumerThreads = kConsumerWarps * 32;
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
  const int c_begin = split * p.rows_per_split;  // < Cmax for every launched split
  const int tile_elems = p.heads * p.dt;
  // A TMA attn box starts at the 4-aligned head at or below h0; the CTA's
  // weights sit a_shift floats into each row of the stage.
  const int a_shift = p.attn_tma ? (h0 & 3) : 0;
  // Stages the producer issues before it knows the sequence length (>= 1,
  // each in its own ring slot, all inside [0, Cmax)).
  const int pre = min(min(min(p.early_stages, p.stages), p.rows_per_split / p.R),
                      (p.Cmax - c_begin + p.R - 1) / p.R);

  uint8_t* vring = smem;
  float* aring = reinterpret_cast<float*>(smem + p.a_off);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.bar_off);
  volatile int& s_flag = *reinterpret_cast<int*>(bars + 2 * kMaxStages);
  const uint32_t full0 = smem_addr(bars);
  const uint32_t empty0 = smem_addr(bars + kMaxStages);

  if (tid == 0) {
    for (int s = 0; s < p.stages; ++s) {
      // expect_tx arrival (+ 32 cp.async arrivals when attn is copied by lanes)
      mbar_init(full0 + 8 * s, p.attn_tma ? 1 : 1 + 32);
      mbar_init(empty0 + 8 * s, kConsumerWarps);  // one arrival per consumer warp
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    s_flag = 0;
  }
  if (warp == kConsumerWarps && lane == 0) {  // kernel parameters: fetch them during the wait
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.v_map)) : "memory");
    if (p.attn_tma)
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.a_map)) : "memory");
  }
  // Producer state that depends on kernel parameters only, ready before the wait.
  const uint64_t policy = evict_first_policy();
  const float* attn_b = p.attn + (size_t)b * p.Cmax * p.Hq + h0;
  const int per_row = p.heads / p.avec;
  const uint32_t vring_s = smem_addr(vring);
  const uint32_t aring_s = smem_addr(aring);
  __syncthreads();

  // Nothing written by earlier kernels is touched before they are done.
  grid_dependency_wait();
  grid_launch_dependents();

  if (warp == kConsumerWarps) {
    // ----------------------------------------------------------------- producer
    // V rows [c0, c0 + R) by TMA (one box, or one box a block of a paged
    // cache); their attn weights by a second TMA box, or (unaligned head
    // groups) the weights of the first `rows` of them by cp.async.
    // Paged: the stage's block indices are loaded by the warp's lanes together
    // (lane j for box j), then lane 0 issues the boxes. Called by all lanes.
    auto load_v = [&](uint32_t dst, int c0, uint32_t full) {
      if (!p.block_table) {
        if (lane == 0) tma_load_4d(dst, &p.v_map, d0, kv_h, c0, b, full, policy);
        return;
      }
      const int nbox = p.R / p.chunk_rows;  // <= 32
      const int2 mine = lane < nbox ? v_row_coord(p, b, c0 + lane * p.chunk_rows) : make_int2(0, 0);
      for (int j = 0; j < nbox; ++j) {
        const int rx = __shfl_sync(0xffffffffu, mine.x, j);
        const int ry = __shfl_sync(0xffffffffu, mine.y, j);
        if (lane == 0)
          tma_load_4d(dst + (uint32_t)(j * p.chunk_rows) * p.dt * 2, &p.v_map, d0, kv_h, rx, ry,
                      full, policy);
      }
    };
    auto issue = [&](int stage, int c0, int rows) {
      const uint32_t full = full0 + 8 * stage;
      if (lane == 0)
        mbar_arrive_expect_tx(full, p.v_stage_bytes + (p.attn_tma ? p.a_stage_bytes : 0u));
      load_v(vring_s + (uint32_t)stage * p.v_stage_bytes, c0, full);
      if (p.attn_tma) {
        if (lane == 0)
          tma_load_3d(aring_s + (uint32_t)stage * p.a_stage_bytes, &p.a_map, h0 - a_shift, c0, b,
                      full, policy);
        return;
      }
      const float* src = attn_b + (size_t)c0 * p.Hq;
      const uint32_t dst = aring_s + 4u * (uint32_t)(stage * p.R * p.ap);
      const int n = rows * per_row;
      for (int i = lane; i < n; i += 32) {
        const int r = i / per_row, k = (i - r * per_row) * p.avec;
        const uint32_t d = dst + 4u * (r * p.ap + k);
        const float* sp = src + (size_t)r * p.Hq + k;
        if (p.avec == 4) cp_async<16>(d, sp);
        else if (p.avec == 2) cp_async<8>(d, sp);
        else cp_async<4>(d, sp);
      }
      cp_async_arrive_noinc(full);
    };
    // The first `pre` stages go out before the sequence length is known
    // (rows past the length are read for nothing, but they lie inside
    // [0, Cmax)); the length load is issued before them and returns while
    // they stream.
    int L = p.seq_lens ? p.seq_lens[b] : p.Cmax;
    issue(0, c_begin, min(p.R, p.Cmax - c_begin));
    for (int it = 1; it < pre; ++it) {
      const int c0 = c_begin + it * p.R;
      issue(it, c0, min(p.R, p.Cmax - c0));
    }
    L = L < 0 ? 0 : (L > p.Cmax ? p.Cmax : L);
    const int nsplit_b = L > 0 ? (L + p.rows_per_split - 1) / p.rows_per_split : 1;
    // Stages the consumers take: none for a split past the context (its
    // consumers leave at once), else every stage holding context (at least
    // one, as the first split of an empty context writes zeros).
    const int c_end = min(c_begin + p.rows_per_split, L);
    const int n_iters =
        split < nsplit_b ? max((c_end - c_begin + p.R - 1) / p.R, 1) : 0;
    int issued = pre;
    bool ok = true;
    for (int it = pre; it < n_iters; ++it) {
      // Self-test: the last stage is never issued (nothing of it is in flight),
      // so the consumers' bounded wait for it runs out.
      if (p.withhold_last && it == n_iters - 1) break;
      const int stage = it % p.stages;
      const uint32_t parity = ((it / p.stages) & 1) ^ 1;
      if (!mbar_wait(empty0 + 8 * stage, parity, p.timeout_ns)) {
        atomicOr(p.status, kErrEmptyWait);
        ok = false;
        break;
      }
      const int c0 = c_begin + it * p.R;
      issue(stage, c0, min(p.R, c_end - c0));
      issued = it + 1;
    }
    cp_async_wait_all();
    if (!ok) {
      // Let every load this CTA issued land before the CTA can exit.
      for (int it = max(0, issued - p.stages); it < issued; ++it)
        if (!mbar_wait(full0 + 8 * (it % p.stages), (it / p.stages) & 1, p.timeout_ns))
          atomicOr(p.status, kErrDrain);
    }
    // Early stages the consumers do not take: let them land before leaving.
    for (int it = n_iters; it < pre; ++it)
      if (!mbar_wait(full0 + 8 * it, 0, p.timeout_ns) && lane == 0) atomicOr(p.status, kErrDrain);
    return;
  }

  // ------------------------------------------------------------------ consumers
  int L = p.seq_lens ? p.seq_lens[b] : p.Cmax;
  L = L < 0 ? 0 : (L > p.Cmax ? p.Cmax : L);
  const int nsplit_b = L > 0 ? (L + p.rows_per_split - 1) / p.rows_per_split : 1;
  if (split >= nsplit_b) return;  // the producer waits for the early stages
  const int c_end = min(c_begin + p.rows_per_split, L);
  const int n_iters = c_end > c_begin ? (c_end - c_begin + p.R - 1) / p.R : 0;
  const int n_stages = max(n_iters, 1);  // stages taken, counting the first one

  const int slots = p.ct * p.nc;
  const int my_col = tid % p.ct;
  const int my_chunk = (tid / p.ct) % p.nc;
  const int my_slot = tid / slots;
  const bool active = my_slot < p.row_par;

  // acc[g][i] holds columns 2i and 2i+1 of head g of the chunk.
  uint64_t acc[GC][4];
#pragma unroll
  for (int g = 0; g < GC; ++g)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[g][i] = 0ull;

  bool ok = true;
  for (int it = 0; it < n_stages; ++it) {
    const int stage = it % p.stages;
    if (!mbar_wait(full0 + 8 * stage, (it / p.stages) & 1, p.full_wait_ns)) {
      atomicOr(p.status, kErrFullWait);
      ok = false;
      break;
    }
    const int rows = min(p.R, c_end - (c_begin + it * p.R));
    const uint16_t* vst =
        reinterpret_cast<const uint16_t*>(vring + (size_t)stage * p.v_stage_bytes) + my_col * 8;
    const float* ast = aring + (size_t)stage * p.R * p.ap + a_shift + my_chunk * GC;
    if (active) {
#pragma unroll 4
      for (int r = my_slot; r < rows; r += p.row_par) {
        const uint4 raw = *reinterpret_cast<const uint4*>(vst + (size_t)r * p.dt);
        float v[8];
        widen8(Tag{}, raw, v);
        uint64_t v2[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) v2[i] = pack2(v[2 * i], v[2 * i + 1]);
        float w[GC];
        load_weights<GC>(ast + (size_t)r * p.ap, w);
#pragma unroll
        for (int g = 0; g < GC; ++g) {
          const uint64_t w2 = pack2(w[g], w[g]);
#pragma unroll
          for (int i = 0; i < 4; ++i) ffma2(acc[g][i], w2, v2[i]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * stage);
  }
  // The ring is reused below: early stages past the context must have landed.
  for (int it = n_stages; it < pre && ok; ++it)
    if (!mbar_wait(full0 + 8 * it, 0, p.timeout_ns)) {
      atomicOr(p.status, kErrFullWait);
      ok = false;
    }
  if (!ok) s_flag = 1;
  consumer_sync<kConsumerThreads>();
  if (s_flag) return;  // the producer drains the loads it issued

  // Row slots -> this CTA's partial: every slot writes its accumulators to its
  // own row of shared memory, then each float4 column is summed over the rows
  // in slot order.
  float* red = reinterpret_cast<float*>(smem);  // the V ring is free now
  if (active) {
    float* dst = red + (size_t)my_slot * tile_elems + (size_t)(my_chunk * GC) * p.dt + my_col * 8;
#pragma unroll
    for (int g = 0; g < GC; ++g) {
      float x[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) unpack2(acc[g][i], x[2 * i], x[2 * i + 1]);
      float4* q = reinterpret_cast<float4*>(dst + (size_t)g * p.dt);
      q[0] = make_float4(x[0], x[1], x[2], x[3]);
      q[1] = make_float4(x[4], x[5], x[6], x[7]);
    }
  }
  consumer_sync<kConsumerThreads>();

  const int ncol4 = tile_elems >> 2;
  const float4* red4 = reinterpret_cast<const float4*>(red);
  float4* part = reinterpret_cast<float4*>(p.ws + ((size_t)tile * p.nsplit + split) * tile_elems);
  for (int col = tid; col < ncol4; col += kConsumerThreads) {
    float4 sum = red4[col];
    sum_strided<false>(sum, red4 + col, ncol4, 1, p.row_par);
    if (nsplit_b == 1) {
      const int e = col * 4, h = e / p.dt, dd = e - h * p.dt;
      *reinterpret_cast<float4*>(p.out + ((size_t)b * p.Hq + h0 + h) * p.D + d0 + dd) = sum;
    } else {
      __stcg(part + col, sum);
    }
  }
}

#ifdef GQA_AV_COMBINE_KERNEL  // defined in exactly one translation unit
// ---------------------------------------------------------------------------
// The split combine. CTA (tile, column block): `parts` threads per float4
// column each sum a fixed chunk of the splits (their loads in flight
// together), then the chunks are added in chunk order. kMode: the partials
// of fixed splits ([tile][split]), of length-balanced splits (one slot a CTA
// of the main kernel), or of the streamed kernel (two slots a CTA: its first
// and its last segment; the tile's partials are those of the CTAs whose
// ranges hold its stages, in CTA order).
// ---------------------------------------------------------------------------
constexpr int kCombineFixed = 0;
constexpr int kCombineBalanced = 1;
constexpr int kCombineStream = 2;

template <int kMode>
__global__ void __launch_bounds__(kCombineThreads)
gqa_av_combine_kernel(const __grid_constant__ CombineParams p) {
  __shared__ float4 chunk_sum[kCombineThreads];
  const int tile = blockIdx.x / p.ctas_per_tile;
  const int blk = blockIdx.x - tile * p.ctas_per_tile;
  const int tiles_per_hg = p.B * p.ndt;
  const int hg = tile / tiles_per_hg;
  const int rem = tile - hg * tiles_per_hg;
  const int b = rem / p.ndt;
  const int dti = rem - b * p.ndt;

  // seq_lens is read before the dependency wait: the main kernel, the only
  // grid this one depends on, does not write it, and the main kernel started
  // (and so could trigger this launch) only after everything before it was
  // done.
  const int ncol4 = p.tile_elems >> 2;
  int nunit;              // splits of the tile
  size_t first, stride;   // float4 offsets of its split 0 and between its splits
  size_t adj0 = 0;        // added to split 0's offset (streamed: a CTA's second slot)
  if constexpr (kMode == kCombineStream) {
    // Tile (b, k): stages [P_b, P_b + n_b) of column k, held by groups g0..g1;
    // group g's CTA is g * K + k, its partial slot 2 (g K + k), except that
    // g0's is its second slot when the tile does not start its range.
    __shared__ longlong2 span;  // (first group, group count)
    __shared__ int first_slot_adj;
    const int K = p.hgroups * p.ndt;
    if (threadIdx.x < 32) {
      const longlong2 r = stream_prefix(p.seq_lens, p.B, p.Cmax, p.R, b);
      const int nb = stream_stages(clamped_len(p.seq_lens, b, p.Cmax), p.R);
      const int Ug0 = p.split_units / K;
      const int Ug = static_cast<int>(r.x < Ug0 ? r.x : Ug0);  // groups that stream
      const int g0 = stream_owner(r.x, r.y, Ug);
      const int g1 = stream_owner(r.x, r.y + nb - 1, Ug);
      if (threadIdx.x == 0) {
        span = make_longlong2(g0, g1 - g0 + 1);
        first_slot_adj = stream_first(r.x, g0, Ug) == r.y ? 0 : 1;
      }
    }
    __syncthreads();
    const size_t k = (size_t)hg * p.ndt + dti;
    nunit = static_cast<int>(span.y);
    first = (size_t)(2 * (span.x * K + k)) * ncol4;
    stride = (size_t)2 * K * ncol4;
    adj0 = (size_t)first_slot_adj * ncol4;
  } else if constexpr (kMode == kCombineBalanced) {
    __shared__ int2 prefix;
    if (threadIdx.x < 32) {
      const int K = p.hgroups * p.ndt;
      const int sps = balanced_sps(p.seq_lens, p.B, p.Cmax, p.R, K, p.split_units);
      const int2 r = balanced_prefix(p.seq_lens, p.Cmax, p.R, sps, b);
      if (threadIdx.x == 0) prefix = r;
    }
    __syncthreads();
    const int K = p.hgroups * p.ndt;
    nunit = prefix.y;
    first = ((size_t)prefix.x * K + hg * p.ndt + dti) * ncol4;
    stride = (size_t)K * ncol4;
  } else {
    int L = p.seq_lens ? p.seq_lens[b] : p.Cmax;
    L = L < 0 ? 0 : (L > p.Cmax ? p.Cmax : L);
    nunit = L > 0 ? (L + p.rows_per_split - 1) / p.rows_per_split : 1;
    first = (size_t)tile * p.nsplit * ncol4;
    stride = ncol4;
  }
  grid_dependency_wait();  // the partials of the main kernel are complete and visible
  grid_launch_dependents();
  if (nunit == 1) return;  // the main kernel wrote this tile's output

  const int t = threadIdx.x;
  const int j = t / p.cols_per_cta;                     // chunk of splits
  const int col = blk * p.cols_per_cta + (t - j * p.cols_per_cta);
  const int chunk = (nunit + p.parts - 1) / p.parts;
  const int lo = j * chunk, hi = min(lo + chunk, nunit);
  const float4* base = reinterpret_cast<const float4*>(p.ws) + first;
  float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
  if (col < ncol4 && lo < hi) {
    sum = __ldcg(base + (size_t)lo * stride + (lo == 0 ? adj0 : 0) + col);
    sum_strided<true>(sum, base + col, stride, lo + 1, hi);
  }
  chunk_sum[t] = sum;
  __syncthreads();
  if (j == 0 && col < ncol4) {
    for (int k = 1; k < p.parts && k * chunk < nunit; ++k) add4(sum, chunk_sum[k * p.cols_per_cta + t]);
    const int e = col * 4, h = e / p.dt, dd = e - h * p.dt;
    *reinterpret_cast<float4*>(p.out + ((size_t)b * p.Hq + hg * p.heads + h) * p.D +
                               dti * p.dt + dd) = sum;
  }
}

#endif  // GQA_AV_COMBINE_KERNEL

// Launch entry points for one (element type, head chunk) instantiation.
template <typename Tag, int GC>
cudaError_t launch(const Params& p, int grid, int smem_bytes, cudaStream_t stream);

template <typename Tag, int GC>
cudaError_t occupancy(int smem_limit, int smem_bytes, int* ctas_per_sm);


cudaError_t launch_combine(const CombineParams& p, int grid, cudaStream_t stream);

}  // namespace gqa_av
