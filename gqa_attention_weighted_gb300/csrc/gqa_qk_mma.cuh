// Decode score step on the 5th-generation tensor cores (tcgen05), sm_103a.
//
// Same operation, tiles, splits and outputs as gqa_qk_kernel (gqa_qk_kernel.cuh):
//   s[b, c, q_h] = scale * sum_d q[b, q_h, d] * K[b, c, q_h / G, d],
// raw scores written to attn, one (max, sum of exp) per head and split for
// gqa_qk_normalize_kernel. Per stage of 128 context rows the CTA computes
//   S[m][n] = sum_k K[c0 + m][k] * Q[n][k]
// as D/16 `tcgen05.mma.cta_group::1.kind::f16` instructions with M = 128 rows,
// N = 2 * Npad (Npad = the group's heads padded to 16), K = D, accumulating in
// fp32 in tensor memory:
//   * A = the K rows, read in place from the TMA stage: D/64 parts of 128 rows
//     x 128 B in the 128-byte swizzle, the K-major SW128 layout (8-row groups
//     1 KiB apart; a K step of 16 advances the start address 32 B within the
//     part, the next part starts 128 x 128 B on).
//   * B = the queries, converted once per CTA: each fp32 q is split into
//     hi = round16(q), lo = round16(q - hi) (bf16 for a bf16 cache, fp16 for
//     fp16; A and B of one MMA have one type), hi rows then lo rows, in the
//     K-major core-matrix layout (8 x 16 B core matrices: 128 B along K,
//     D/8 x 128 B between 8-row groups). One MMA pass gives both products:
//     K is exact in its type and 16-bit x 16-bit products are exact in fp32.
//   * D is double-buffered in tensor memory (2 x 2 Npad columns). The four
//     accumulator warps (warp w reads lanes 32w..32w+31, one context row a
//     thread) read a stage's D with tcgen05.ld, add hi + lo, scale, write the
//     row's scores and update a running (max, sum of exp) per head.
// Warps: 0-3 accumulate (and convert the queries first), 4 is the TMA
// producer, 5 allocates tensor memory and one of its threads issues the MMAs.
// Every mbarrier wait is bounded; on expiry the CTA sets the device status
// word, lets its copies and MMAs in flight finish, frees its tensor memory and
// returns.
#pragma once

#include "gqa_av_mma.cuh"
#include "gqa_qk_kernel.cuh"

namespace gqa_av {

constexpr int kQkMmaRows = 128;                        // context rows per stage (M)
constexpr int kQkMmaThreads = 32 * (kMmaAccWarps + 2);  // + producer and MMA warps

// Instruction descriptor of kind::f16: fp32 D, A and B of one 16-bit type,
// both K-major, N x M = n x 128.
template <typename Tag>
__host__ __device__ constexpr uint32_t qk_mma_idesc(int n) {
  return (1u << 4) | (std::is_same<Tag, Bf16Tag>::value ? ((1u << 7) | (1u << 10)) : 0u) |
         (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(kQkMmaRows >> 4) << 24);
}

// A query pair split into 16-bit hi and lo halves (unscaled: queries are
// O(1), unlike the AV kernel's weights).
__device__ __forceinline__ void split_query(Bf16Tag t, float a, float b, uint32_t& hi,
                                            uint32_t& lo) {
  split_weights(t, a, b, hi, lo);
}
__device__ __forceinline__ void split_query(Fp16Tag, float a, float b, uint32_t& hi,
                                            uint32_t& lo) {
  const __half2 h = __floats2half2_rn(a, b);
  const float2 hf = __half22float2(h);
  const __half2 l = __floats2half2_rn(a - hf.x, b - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// The queries of `heads` consecutive heads (row n at q_rows + n * 8 * nkc)
// -> the B operand's hi and lo rows, element (n, k) at ((n / 8) * nkc + k / 8)
// * 128 + (n % 8) * 16 + (k % 8) * 2; rows n >= heads are zero. A thread takes
// items t = first, first + stride, ... (item t: row t % N, 8 columns from
// 8 (t / N)) and issues the loads of BATCH items before converting any, so
// the operand costs about one round of global loads per batch (one item a
// round made the first MMA of an MQA-shaped call wait 4 us for its queries).
// load_queries issues one batch (items t0, t0 + stride, ... into x),
// store_queries converts and stores it; convert_queries does every batch.
template <int N, int BATCH>
__device__ __forceinline__ void load_queries(const float* q_rows, int heads, int nkc, int t0,
                                             int stride, float4 (&x)[BATCH][2]) {
  const int items = N * nkc;
#pragma unroll
  for (int u = 0; u < BATCH; ++u) {
    const int t = t0 + u * stride;
    const int n = t % N, kc = t / N;
    if (t < items && n < heads) {
      const float4* src = reinterpret_cast<const float4*>(q_rows + (size_t)n * nkc * 8 + kc * 8);
      x[u][0] = src[0];
      x[u][1] = src[1];
    } else {
      x[u][0] = x[u][1] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
  }
}

template <typename Tag, int N, int BATCH>
__device__ __forceinline__ void store_queries(const float4 (&x)[BATCH][2], int nkc, uint8_t* bst,
                                              uint32_t b_half, int t0, int stride) {
  const int items = N * nkc;
#pragma unroll
  for (int u = 0; u < BATCH; ++u) {
    const int t = t0 + u * stride;
    if (t < items) {
      const int n = t % N, kc = t / N;
      uint32_t hi[4], lo[4];
      split_query(Tag{}, x[u][0].x, x[u][0].y, hi[0], lo[0]);
      split_query(Tag{}, x[u][0].z, x[u][0].w, hi[1], lo[1]);
      split_query(Tag{}, x[u][1].x, x[u][1].y, hi[2], lo[2]);
      split_query(Tag{}, x[u][1].z, x[u][1].w, hi[3], lo[3]);
      const size_t off = (size_t)((n >> 3) * nkc + kc) * 128 + (n & 7) * 16;
      *reinterpret_cast<uint4*>(bst + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(bst + b_half + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
  }
}

template <typename Tag, int N, int BATCH>
__device__ __forceinline__ void convert_queries(const float* q_rows, int heads, int nkc,
                                                uint8_t* bst, uint32_t b_half, int first,
                                                int stride) {
  for (int t0 = first; t0 < N * nkc; t0 += BATCH * stride) {
    float4 x[BATCH][2];
    load_queries<N, BATCH>(q_rows, heads, nkc, t0, stride, x);
    store_queries<Tag, N, BATCH>(x, nkc, bst, b_half, t0, stride);
  }
}

// One row's scores into a thread's running (max, sum of exp(x - max)) per
// head, without branches on the data: max first, the old sum rescaled to it
// (by exactly 1 when the max did not move), plus exp(s - max). Heads go in
// groups of four (a group past `heads` is skipped; padding inside the last
// group is updated and never read). A data-dependent branch per head made
// the lanes of a warp diverge on every row: with 16 heads the accumulators
// took 1.7 us a 128-row stage and bounded the streamed kernel.
template <int N>
__device__ __forceinline__ void online_lse_update(float (&mx)[N], float (&sm)[N],
                                                  const float (&s)[N], int heads) {
#pragma unroll
  for (int n0 = 0; n0 < N; n0 += 4) {
    if (n0 < heads) {
#pragma unroll
      for (int n = n0; n < n0 + 4; ++n) {
        const float mn = fmaxf(mx[n], s[n]);
        const float keep = mn == mx[n] ? 1.0f : __expf(mx[n] - mn);
        sm[n] = sm[n] * keep + __expf(s[n] - mn);
        mx[n] = mn;
      }
    }
  }
}

// The (max, sum of exp(x - max)) over a warp's lanes of each of the first
// `heads` of N running pairs, four heads at a time so that their shuffles
// overlap; lane 0 writes head n's pair to red[n]. Deterministic (fixed
// butterflies): the maximum first, then each lane's sum rescaled to it.
template <int N>
__device__ __forceinline__ void warp_lse_heads(const float (&mx)[N], const float (&sm)[N],
                                               int heads, float2* red) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int n0 = 0; n0 < N; n0 += 4) {
    if (n0 < heads) {
      float M[4], S[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) M[i] = mx[n0 + i];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int i = 0; i < 4; ++i) M[i] = fmaxf(M[i], __shfl_xor_sync(0xffffffffu, M[i], o));
#pragma unroll
      for (int i = 0; i < 4; ++i)
        S[i] = mx[n0 + i] == -INFINITY ? 0.0f : sm[n0 + i] * __expf(mx[n0 + i] - M[i]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int i = 0; i < 4; ++i) S[i] += __shfl_xor_sync(0xffffffffu, S[i], o);
      if (lane == 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (n0 + i < heads) red[n0 + i] = make_float2(M[i], S[i]);
      }
    }
  }
}

// Shared memory (offsets from a 1024-byte-aligned base):
//   [K ring: stages x D/64 parts x 128 rows x 128 B]   (stage_bytes each)
//   [B: 2 Npad rows x D columns, 16-bit, core-matrix layout]   at b_off
//   [reduction: 4 warps x Npad float2]                         at red_off
//   [mbarriers: full, empty (kMaxStages each), dfull[2], dfree[2], qready, drain] at bar_off
//   [tensor-memory address]
template <typename Tag, int NB>
__global__ void __launch_bounds__(kQkMmaThreads, 1)
    gqa_qk_mma_kernel(const __grid_constant__ QkParams p) {
  constexpr int N = 16 * NB;  // Npad
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_addr(smem_raw);
  const uint32_t base_s = (raw_s + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base_s - raw_s);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  constexpr int producer_warp = kMmaAccWarps;
  constexpr int issuer_warp = kMmaAccWarps + 1;

  const int tile = blockIdx.x / p.nsplit;
  const int split = blockIdx.x - tile * p.nsplit;
  const int hg = tile / p.B;
  const int b = tile - hg * p.B;
  const int h0 = hg * p.heads;
  const int kv_h = h0 / p.G;
  const int c_begin = split * p.rows_per_split;
  const int pre = min(min(p.stages, p.rows_per_split / kQkMmaRows),
                      (p.Cmax - c_begin + kQkMmaRows - 1) / kQkMmaRows);

  float2* red = reinterpret_cast<float2*>(smem + p.red_off);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.bar_off);
  const uint32_t full0 = smem_addr(bars);
  const uint32_t empty0 = smem_addr(bars + kMaxStages);
  const uint32_t dfull0 = smem_addr(bars + 2 * kMaxStages);
  const uint32_t dfree0 = smem_addr(bars + 2 * kMaxStages + 2);
  const uint32_t qready = smem_addr(bars + 2 * kMaxStages + 4);
  const uint32_t drain = smem_addr(bars + 2 * kMaxStages + 5);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kMaxStages + 6);

  if (warp == issuer_warp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tmem_slot)),
                 "r"(p.tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);  // one tcgen05.commit per stage
    }
    for (int j = 0; j < 2; ++j) {
      mbar_init(dfull0 + 8 * j, 1);
      mbar_init(dfree0 + 8 * j, kMmaAccWarps);
    }
    mbar_init(qready, kMmaAccWarps);
    mbar_init(drain, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == producer_warp && lane == 0)
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.k_map)) : "memory");
  const uint64_t policy = evict_first_policy();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  grid_dependency_wait();
  grid_launch_dependents();

  // The first stages do not depend on the length: the producer issues them
  // before its load of seq_lens (measured: the load delayed the first copy
  // by about 0.8 us).
  auto issue = [&](int stage, int c0) {
    if (lane == 0) {
      const uint32_t full = full0 + 8 * stage;
      mbar_arrive_expect_tx(full, p.stage_bytes);
      const uint32_t dst = base_s + (uint32_t)stage * p.stage_bytes;
      for (int part = 0; part < p.parts; ++part)
        tma_load_4d(dst + (uint32_t)part * kQkMmaRows * 128, &p.k_map, 64 * part, kv_h, c0, b,
                    full, policy);
    }
  };
  if (warp == producer_warp)
    for (int it = 0; it < pre; ++it) issue(it, c_begin + it * kQkMmaRows);

  const int L = clamped_len(p.seq_lens, b, p.Cmax);
  const int nsplit_b = L > 0 ? (L + p.rows_per_split - 1) / p.rows_per_split : 1;
  const int c_end = min(c_begin + p.rows_per_split, L);
  const int n_iters =
      split < nsplit_b && c_end > c_begin ? (c_end - c_begin + kQkMmaRows - 1) / kQkMmaRows : 0;

  if (warp == producer_warp) {
    // ----------------------------------------------------------------- producer
    bool ok = true;
    int issued = pre;
    for (int it = pre; it < n_iters; ++it) {
      const int stage = it % p.stages;
      if (!mbar_wait(empty0 + 8 * stage, ((it / p.stages) & 1) ^ 1, p.timeout_ns)) {
        if (lane == 0) atomicOr(p.status, kErrEmptyWait);
        ok = false;
        break;
      }
      issue(stage, c_begin + it * kQkMmaRows);
      issued = it + 1;
    }
    if (!ok) {
      for (int it = max(0, issued - p.stages); it < issued; ++it)
        if (!mbar_wait(full0 + 8 * (it % p.stages), (it / p.stages) & 1, p.timeout_ns) && lane == 0)
          atomicOr(p.status, kErrDrain);
    }
    for (int it = n_iters; it < pre; ++it)
      if (!mbar_wait(full0 + 8 * it, 0, p.timeout_ns) && lane == 0) atomicOr(p.status, kErrDrain);
    return;
  }

  const int nkc = p.D / 8;                          // 16-byte core-matrix columns along K
  const uint32_t b_half = (uint32_t)N * p.D * 2;    // bytes of the hi (or lo) rows

  if (warp == issuer_warp) {
    // -------------------------------------------------------------- MMA issuer
    bool ok = true;
    if (lane == 0) {
      const uint32_t idesc = qk_mma_idesc<Tag>(2 * N);
      const uint32_t bb = base_s + p.b_off;
      const uint64_t bd0 = smem_desc(bb, 128, (uint32_t)nkc * 128, 0);
      int issued = 0;
      if (n_iters > 0 && !mbar_poll(qready, 0, p.timeout_ns)) {
        atomicOr(p.status, kErrMmaWait);
        ok = false;
      }
      for (int it = 0; ok && it < n_iters; ++it) {
        const int stage = it % p.stages, j = it & 1;
        if (!mbar_poll(full0 + 8 * stage, (it / p.stages) & 1, p.timeout_ns) ||
            (it >= 2 && !mbar_poll(dfree0 + 8 * j, ((it - 2) >> 1) & 1, p.timeout_ns))) {
          atomicOr(p.status, kErrMmaWait);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(j * 2 * N);
        const uint32_t a0 = base_s + (uint32_t)stage * p.stage_bytes;
        for (int kk = 0; kk < p.D / 16; ++kk) {
          // K step kk: part kk / 4 (128 x 128 B each), 32 B into it per step.
          const uint32_t a_addr = a0 + (uint32_t)(kk >> 2) * kQkMmaRows * 128 + (uint32_t)(kk & 3) * 32;
          const uint64_t ad = smem_desc(a_addr, 16, 1024, 2);
          mma_f16(d_tmem, ad, bd0 + (uint64_t)(kk * (256 >> 4)), idesc, kk > 0 ? 1u : 0u);
        }
        mma_commit(empty0 + 8 * stage);  // the K slot is free once these MMAs are done
        mma_commit(dfull0 + 8 * j);
        issued = it + 1;
      }
      if (issued > 0) {
        mma_commit(drain);
        if (!mbar_wait(drain, 0, p.timeout_ns)) atomicOr(p.status, kErrMmaWait);
      }
    }
    __syncwarp();
    (void)ok;
    mma_team_sync();  // the accumulators are done with tensor memory
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(p.tmem_cols)
                 : "memory");
    return;
  }

  // -------------------------------------------------------------- accumulators
  // The group's queries -> B hi / lo (element (n, k) at ((n / 8) * nkc + k / 8)
  // * 128 + (n % 8) * 16 + (k % 8) * 2; heads past the group are zero).
  {
    convert_queries<Tag, N, 4>(p.q + ((size_t)b * p.Hq + h0) * p.D, p.heads, nkc, smem + p.b_off,
                               b_half, tid, 32 * kMmaAccWarps);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) mbar_arrive(qready);
  }

  const int m_row = tid;  // tensor-memory lane = context row of the stage
  float mx[N], sm[N];
#pragma unroll
  for (int n = 0; n < N; ++n) {
    mx[n] = -INFINITY;
    sm[n] = 0.0f;
  }
  bool ok = true;
  for (int it = 0; it < n_iters; ++it) {
    const int j = it & 1;
    if (!mbar_wait(dfull0 + 8 * j, (it >> 1) & 1, p.timeout_ns)) {
      atomicOr(p.status, kErrMmaWait);
      ok = false;
      break;
    }
    tc_fence_after();
    const uint32_t taddr = tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)(j * 2 * N);
    float s[N];
#pragma unroll
    for (int q = 0; q < NB; ++q) {
      float h[16], l[16];
      tmem_ld16(taddr + 16u * q, h);
      tmem_ld16(taddr + (uint32_t)N + 16u * q, l);
#pragma unroll
      for (int i = 0; i < 16; ++i) s[16 * q + i] = (h[i] + l[i]) * p.scale;
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(dfree0 + 8 * j);
    const int c = c_begin + it * kQkMmaRows + m_row;
    if (c < c_end) {
      float* dst = p.attn + ((size_t)b * p.Cmax + c) * p.Hq + h0;
      // 16-byte stores where the group's heads allow (attn rows are 16-byte
      // aligned, and so is head h0 of a group of a multiple of 4 heads).
      if (p.heads % 4 == 0 && p.Hq % 4 == 0) {
#pragma unroll
        for (int n = 0; n < N; n += 4)
          if (n < p.heads)
            __stcg(reinterpret_cast<float4*>(dst + n), make_float4(s[n], s[n + 1], s[n + 2], s[n + 3]));
      } else {
#pragma unroll
        for (int n = 0; n < N; ++n)
          if (n < p.heads) dst[n] = s[n];
      }
      online_lse_update<N>(mx, sm, s, p.heads);
    }
  }

  // One (max, sum) per head of the group (not the padding up to N) for the
  // split: over each warp's lanes, then over the four warps in warp order.
  warp_lse_heads<N>(mx, sm, p.heads, red + (size_t)warp * N);
  named_sync(1, 32 * kMmaAccWarps);
  if (tid < p.heads && ok && n_iters > 0)
    p.stats[((size_t)tile * p.nsplit + split) * p.heads + tid] = lse_of(red + tid, kMmaAccWarps, N);
  tc_fence_before();
  mma_team_sync();
}

}  // namespace gqa_av
