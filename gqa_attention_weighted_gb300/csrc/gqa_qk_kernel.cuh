// Decode score step for sm_103a (GB300): scaled query-key products and the
// softmax over the context that gives the AV reduction its weights.
//
//   s[b, c, q_h]    = scale * sum_d q[b, q_h, d] * K[b, c, q_h / G, d]
//   attn[b, c, q_h] = exp(s - max_c s) / sum_c exp(s - max_c s),  c < L_b.
//
// This is the step before the AV coop-GEMV of LLM decode (page "pytorch/
// executorch pull 21063", summary paragraph) with the same query-to-KV-head
// mapping, so each K row is read from HBM once for all G query heads of its
// group, as V is there.
//
// gqa_qk_kernel: one CTA owns a tile (head group, b) and a context split of
// it. A producer warp streams K rows by TMA into a shared-memory ring, as
// D / 64 boxes of 64 columns in the 128-byte swizzle, so that the consumer
// threads, one K row each, read their 16-byte chunks without bank conflicts.
// The group's query vectors sit in shared memory and are read as warp-wide
// broadcasts. Each consumer thread owns one row of a stage and a chunk of GC
// heads: it writes the GC raw scores of its row to attn and keeps a running
// (max, sum of exp) per head; the CTA reduces these to one (max, sum) per
// head for its split.
//
// gqa_qk_normalize_kernel (launched next, programmatic dependent launch):
// combines the splits' (max, sum) pairs of each (b, q_h) (M the largest max,
// S the sum of each split's sum rescaled to M, both in a fixed order) and
// rewrites attn[b, c, :] = exp(s - M) / S for the in-range rows. Entries at
// c >= L_b are never written. Results are bitwise reproducible for a fixed
// launch shape.
#pragma once

#include <type_traits>

#include "gqa_av_kernel.cuh"

namespace gqa_av {

constexpr int kQkConsumerWarps = 8;
constexpr int kQkConsumerThreads = 32 * kQkConsumerWarps;
constexpr int kQkThreads = kQkConsumerThreads + 32;  // + the producer warp
constexpr int kQkNormThreads = 256;
constexpr int kQkNormBatch = 8;          // scores each normalise thread loads at once
constexpr int kQkNormMaxPairs = 3072;     // (head, split) pairs staged in shared memory
constexpr int kQkNormCtasPerSm = 4;       // normalise CTAs resident an SM (their registers)
constexpr int kQkNormMaxIters = 8;        // batches of scores a normalise CTA rewrites, at most
constexpr int kQkNormFastSeg = 32;        // pairs a head a thread merges on its own, at most
// Floats a normalise load moves: 4 when Hq % 4 == 0 (every row then starts on
// a 16-byte boundary), else 1; loads a thread has in flight per batch.
__host__ __device__ constexpr int qk_norm_vec(int Hq) { return Hq % 4 == 0 ? 4 : 1; }
__host__ __device__ constexpr int qk_norm_loads(int vec) { return vec == 4 ? 4 : 8; }
// Rows a normalise CTA rewrites per batch. With Hq / vec <= kQkNormThreads
// vectors a row, a thread keeps one column of vectors (fixed heads) over
// kQkNormThreads / (Hq / vec) rows a pass; wider rows go element by element.
__host__ __device__ constexpr int qk_norm_rows_per_batch(int Hq) {
  return Hq / qk_norm_vec(Hq) <= kQkNormThreads
             ? qk_norm_loads(qk_norm_vec(Hq)) * (kQkNormThreads / (Hq / qk_norm_vec(Hq)))
             : (qk_norm_loads(qk_norm_vec(Hq)) * qk_norm_vec(Hq) * kQkNormThreads + Hq - 1) / Hq;
}
constexpr int kQkMaxHeads = 64;

struct alignas(64) QkParams {
  CUtensorMap k_map;            // K as 4-D {D, Hkv, Cmax, B}; box {64, 1, R, 1}, 128B swizzle
  const float* q;               // [B, Hq, D]
  const int32_t* seq_lens;      // [B] or null
  float* attn;                  // [B, Cmax, Hq]
  float2* stats;                // [tiles][nsplit][heads] (max, sum of exp) per split
  unsigned int* status;         // device status word
  float scale;
  int B, Cmax, Hq, Hkv, D, G;
  int heads;                    // query heads per CTA (G, or 1 per head)
  int hgroups;                  // Hq / heads
  int nc;                       // heads / GC head chunks
  int rs;                       // consumer threads per head chunk (256 / nc, a multiple of 32)
  int R;                        // K rows per stage (<= rs; thread r of a chunk takes row r)
  int stages;
  int rows_per_split, nsplit;
  int parts;                    // D / 64 boxes per row
  uint32_t stage_bytes;         // R * D * 2
  uint32_t q_off, red_off, bar_off;  // shared-memory offsets from the 1024-aligned base
  long long timeout_ns;
  // Tensor-core kernels only.
  uint32_t b_off;               // shared-memory offset of the B (query hi / lo) operand
  uint32_t tmem_cols;           // tensor-memory columns allocated (power of 2 >= 4 x Npad)
  // Streamed kernel only: CTAs (groups of hgroups), lengths in shared memory,
  // the (max, sum) of each tile one CTA held whole [B][hgroups][heads].
  int split_units;
  uint32_t lens_off;
  float2* stats_whole;
};

struct QkNormParams {
  const float2* stats;          // as QkParams::stats
  const int32_t* seq_lens;
  float* attn;
  int B, Cmax, Hq, heads, hgroups, rows_per_split, nsplit;
  int rows_per_cta;             // context rows each CTA rewrites
  int ctas_per_b;
  int split_units;              // streamed kernel: its CTAs
  const float2* stats_whole;    // streamed kernel: as QkParams::stats_whole
};

// Merge of two (max, sum of exp(x - max)) pairs.
__device__ __forceinline__ void lse_merge(float& m, float& l, float m2, float l2) {
  const float mn = fmaxf(m, m2);
  const float a = m == -INFINITY ? 0.0f : l * __expf(m - mn);
  const float b = m2 == -INFINITY ? 0.0f : l2 * __expf(m2 - mn);
  m = mn;
  l = a + b;
}

// The (max, sum of exp(x - max)) of `n` pairs in memory (stride apart): the
// maximum first, then every pair's sum rescaled to it, added in index order.
__device__ __forceinline__ float2 lse_of(const float2* v, int n, int stride) {
  float M = -INFINITY, S = 0.0f;
  for (int i = 0; i < n; ++i) M = fmaxf(M, v[(size_t)i * stride].x);
  for (int i = 0; i < n; ++i) {
    const float2 x = v[(size_t)i * stride];
    if (x.x != -INFINITY) S += x.y * __expf(x.x - M);
  }
  return make_float2(M, S);
}

// ---------------------------------------------------------------------------
// Shared memory (offsets from a 1024-byte-aligned base):
//   [K ring: stages x parts x R x 128 B, each part in the 128-byte swizzle]
//   [q: heads x D floats]
//   [reduction: kQkConsumerWarps x GC float2]
//   [mbarriers: full, empty (kMaxStages each)]
template <typename Tag, int GC>
__global__ void __launch_bounds__(kQkThreads, 1) gqa_qk_kernel(const __grid_constant__ QkParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_addr(smem_raw);
  const uint32_t base_s = (raw_s + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base_s - raw_s);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  const int tile = blockIdx.x / p.nsplit;
  const int split = blockIdx.x - tile * p.nsplit;
  const int hg = tile / p.B;
  const int b = tile - hg * p.B;
  const int h0 = hg * p.heads;
  const int kv_h = h0 / p.G;
  const int c_begin = split * p.rows_per_split;
  const int pre = min(min(p.stages, p.rows_per_split / p.R), (p.Cmax - c_begin + p.R - 1) / p.R);

  float* q_s = reinterpret_cast<float*>(smem + p.q_off);
  float2* red = reinterpret_cast<float2*>(smem + p.red_off);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.bar_off);
  const uint32_t full0 = smem_addr(bars);
  const uint32_t empty0 = smem_addr(bars + kMaxStages);

  if (tid == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kQkConsumerWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kQkConsumerWarps && lane == 0)
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.k_map)) : "memory");
  const uint64_t policy = evict_first_policy();
  __syncthreads();

  grid_dependency_wait();
  grid_launch_dependents();

  const int L = clamped_len(p.seq_lens, b, p.Cmax);
  const int nsplit_b = L > 0 ? (L + p.rows_per_split - 1) / p.rows_per_split : 1;
  const int c_end = min(c_begin + p.rows_per_split, L);
  const int n_iters = split < nsplit_b && c_end > c_begin ? (c_end - c_begin + p.R - 1) / p.R : 0;

  if (warp == kQkConsumerWarps) {
    // ----------------------------------------------------------------- producer
    auto issue = [&](int stage, int c0) {
      if (lane == 0) {
        const uint32_t full = full0 + 8 * stage;
        mbar_arrive_expect_tx(full, p.stage_bytes);
        const uint32_t dst = base_s + (uint32_t)stage * p.stage_bytes;
        for (int part = 0; part < p.parts; ++part)
          tma_load_4d(dst + (uint32_t)part * p.R * 128, &p.k_map, 64 * part, kv_h, c0, b, full,
                      policy);
      }
    };
    for (int it = 0; it < pre; ++it) issue(it, c_begin + it * p.R);  // before the length is known
    bool ok = true;
    int issued = pre;
    for (int it = pre; it < n_iters; ++it) {
      const int stage = it % p.stages;
      if (!mbar_wait(empty0 + 8 * stage, ((it / p.stages) & 1) ^ 1, p.timeout_ns)) {
        if (lane == 0) atomicOr(p.status, kErrEmptyWait);
        ok = false;
        break;
      }
      issue(stage, c_begin + it * p.R);
      issued = it + 1;
    }
    if (!ok) {
      for (int it = max(0, issued - p.stages); it < issued; ++it)
        if (!mbar_wait(full0 + 8 * (it % p.stages), (it / p.stages) & 1, p.timeout_ns) && lane == 0)
          atomicOr(p.status, kErrDrain);
    }
    // Early stages past the split's rows: let them land before the CTA exits.
    for (int it = n_iters; it < pre; ++it)
      if (!mbar_wait(full0 + 8 * it, 0, p.timeout_ns) && lane == 0) atomicOr(p.status, kErrDrain);
    return;
  }

  // ---------------------------------------------------------------- consumers
  // The group's query vectors into shared memory (read as broadcasts below).
  {
    const float4* src = reinterpret_cast<const float4*>(p.q + ((size_t)b * p.Hq + h0) * p.D);
    float4* dst = reinterpret_cast<float4*>(q_s);
    for (int i = tid; i < p.heads * p.D / 4; i += kQkConsumerThreads) dst[i] = src[i];
  }
  named_sync(1, kQkConsumerThreads);

  const int hc = tid / p.rs;         // head chunk
  const int r = tid - hc * p.rs;     // row of each stage
  const bool active = hc < p.nc && r < p.R;
  const float* qh = q_s + (size_t)(hc * GC) * p.D;
  float m[GC], l[GC];
#pragma unroll
  for (int g = 0; g < GC; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.0f;
  }
  bool ok = true;
  for (int it = 0; it < n_iters; ++it) {
    const int stage = it % p.stages;
    if (!mbar_wait(full0 + 8 * stage, (it / p.stages) & 1, p.timeout_ns)) {
      atomicOr(p.status, kErrFullWait);
      ok = false;
      break;
    }
    const int c = c_begin + it * p.R + r;
    if (active && c < c_end) {
      const uint8_t* row = smem + (size_t)stage * p.stage_bytes + (size_t)r * 128;
      float dot[GC];
#pragma unroll
      for (int g = 0; g < GC; ++g) dot[g] = 0.0f;
      for (int part = 0; part < p.parts; ++part) {
        const uint8_t* prow = row + (size_t)part * p.R * 128;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          // 16-byte chunk j of this 64-column part, where the swizzle put it.
          const uint4 raw = *reinterpret_cast<const uint4*>(prow + ((j ^ (r & 7)) << 4));
          float kf[8];
          widen8(Tag{}, raw, kf);
          const int d = part * 64 + j * 8;
#pragma unroll
          for (int g = 0; g < GC; ++g) {
            const float4 qa = *reinterpret_cast<const float4*>(qh + (size_t)g * p.D + d);
            const float4 qb = *reinterpret_cast<const float4*>(qh + (size_t)g * p.D + d + 4);
            float acc = dot[g];
            acc = fmaf(kf[0], qa.x, acc);
            acc = fmaf(kf[1], qa.y, acc);
            acc = fmaf(kf[2], qa.z, acc);
            acc = fmaf(kf[3], qa.w, acc);
            acc = fmaf(kf[4], qb.x, acc);
            acc = fmaf(kf[5], qb.y, acc);
            acc = fmaf(kf[6], qb.z, acc);
            acc = fmaf(kf[7], qb.w, acc);
            dot[g] = acc;
          }
        }
      }
      float* dst = p.attn + ((size_t)b * p.Cmax + c) * p.Hq + h0 + hc * GC;
#pragma unroll
      for (int g = 0; g < GC; ++g) {
        const float s = dot[g] * p.scale;
        dst[g] = s;
        if (s > m[g]) {
          l[g] = (m[g] == -INFINITY ? 0.0f : l[g] * __expf(m[g] - s)) + 1.0f;
          m[g] = s;
        } else {
          l[g] += __expf(s - m[g]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * stage);
  }

  // One (max, sum) per head for the split: within each warp (rs is a multiple
  // of 32, so a warp's lanes share one head chunk), then over the chunk's
  // warps in warp order.
#pragma unroll
  for (int g = 0; g < GC; ++g) {
    float mm = m[g], ll = l[g];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, mm, o);
      const float l2 = __shfl_xor_sync(0xffffffffu, ll, o);
      lse_merge(mm, ll, m2, l2);
    }
    if (lane == 0) red[(size_t)warp * GC + g] = make_float2(mm, ll);  // (-inf, 0) if no rows
  }
  named_sync(1, kQkConsumerThreads);
  if (tid < p.heads && ok && n_iters > 0) {
    const int chunk = tid / GC, g = tid - chunk * GC;
    const int wpc = p.rs / 32;  // warps per head chunk
    float mm = -INFINITY, ll = 0.0f;
    for (int w = chunk * wpc; w < (chunk + 1) * wpc; ++w) {
      const float2 v = red[(size_t)w * GC + g];
      lse_merge(mm, ll, v.x, v.y);
    }
    p.stats[((size_t)tile * p.nsplit + split) * p.heads + tid] = make_float2(mm, ll);
  }
}

// ---------------------------------------------------------------------------
// The normalise step of one CTA (sequence b, rows [c0, c1)), shared by the
// fixed-split and streamed score kernels: every head of b has `nseg` (max,
// sum) pairs, pair (h, i) at slot(h / heads, i)[h % heads] (the heads of one
// slot contiguous). The routine waits for the score kernel (programmatic
// dependent launch) after working out what needs no results of it, then:
//   1. loads the first batch of the block's scores into registers (a batch
//      is qk_norm_rows_per_batch(Hq) rows, a few loads a thread) and every
//      pair into shared memory (a slot's heads are adjacent addresses), all
//      in flight together;
//   2. per head M = max_i m_i, then S = sum_i l_i exp(m_i - M): with at most
//      kQkNormFastSeg segments by the head's own thread in segment order,
//      else with `tph` threads a head (a power of two up to 32) taking
//      segments part, part + tph, ... and fixed butterflies over them (each
//      dependent step of a merge costs about 0.2 us, so few segments go
//      without the butterflies);
//   3. attn = exp(s - M) / S, batch after batch, the next batch's loads
//      issued before the current one is written.
// ---------------------------------------------------------------------------
template <int VEC, typename Slot>
__device__ __forceinline__ void qk_normalize_rows(float* attn_b, int Hq, int heads, int nseg,
                                                  int c0, int c1, Slot slot, float2* ms,
                                                  float2* pairs) {
  // VEC floats a load, kLoads loads a thread a batch. Rows of at most
  // kQkNormThreads vectors: thread t takes vector column t % cols of rows
  // t / cols, t / cols + rpp, ... (rpp rows a pass), so its heads, and their
  // (M, 1 / S), are the same for every row it writes. Wider rows: element
  // index base + (t + u kQkNormThreads) VEC of the block.
  constexpr int kLoads = qk_norm_loads(VEC);
  using Vec = typename std::conditional<VEC == 4, float4, float>::type;
  const int tid = threadIdx.x;
  const int rows = c1 - c0;
  const int n = rows * Hq;
  float* row0 = attn_b + (size_t)c0 * Hq;
  const int cols = Hq / VEC;
  const bool by_col = cols <= kQkNormThreads;
  const int rpp = by_col ? kQkNormThreads / cols : 0;
  const int my_col = by_col ? tid % cols : 0;
  const int my_row = by_col ? tid / cols : 0;
  const bool active = by_col && my_row < rpp;
  const int rpb = kLoads * rpp;              // rows a batch (by column)
  constexpr int kChunk = kLoads * VEC * kQkNormThreads;  // elements a batch (wide rows)
  auto load = [&](Vec (&x)[kLoads], int base) {  // base: first row, or first element
#pragma unroll
    for (int u = 0; u < kLoads; ++u) {
      if (by_col) {
        const int r = base + u * rpp + my_row;
        if (active && r < rows)
          x[u] = __ldcg(reinterpret_cast<const Vec*>(row0 + (size_t)r * Hq + my_col * VEC));
      } else {
        const int i = base + (tid + u * kQkNormThreads) * VEC;
        if (i < n) x[u] = __ldcg(reinterpret_cast<const Vec*>(row0 + i));
      }
    }
  };
  // Pair i of the staging order (i = (k * nseg + seg) * heads + hh) comes
  // from slot(k, seg)[hh]. When all pairs fit one batch of loads (the usual
  // case), each thread works out the addresses of its pairs before the
  // dependency wait, so the loads issue as soon as it returns.
  const int per_k = nseg * heads;
  const int npairs = Hq * nseg;
  const bool staged = npairs <= kQkNormMaxPairs;
  const bool one_batch = npairs <= kQkNormBatch * kQkNormThreads;
  const float2* src[kQkNormBatch];
#pragma unroll
  for (int u = 0; u < kQkNormBatch; ++u) {
    const int i = tid + u * kQkNormThreads;
    src[u] = nullptr;
    if (one_batch && i < npairs) {
      const int k = i / per_k, r = i - k * per_k;
      const int seg = r / heads;
      src[u] = slot(k, seg) + (r - seg * heads);
    }
  }
  grid_dependency_wait();  // scores and pairs of the score kernel are visible
  grid_launch_dependents();
  Vec x[kLoads];
  load(x, 0);
  if (one_batch) {
    float2 v[kQkNormBatch];
#pragma unroll
    for (int u = 0; u < kQkNormBatch; ++u)
      if (src[u]) v[u] = __ldcg(src[u]);
#pragma unroll
    for (int u = 0; u < kQkNormBatch; ++u)
      if (src[u]) pairs[tid + u * kQkNormThreads] = v[u];
  } else if (staged) {
    for (int i0 = tid; i0 < npairs; i0 += kQkNormBatch * kQkNormThreads) {
      float2 v[kQkNormBatch];
#pragma unroll
      for (int u = 0; u < kQkNormBatch; ++u) {
        const int i = i0 + u * kQkNormThreads;
        if (i < npairs) {
          const int k = i / per_k, r = i - k * per_k;
          const int seg = r / heads;
          v[u] = __ldcg(slot(k, seg) + (r - seg * heads));
        }
      }
#pragma unroll
      for (int u = 0; u < kQkNormBatch; ++u) {
        const int i = i0 + u * kQkNormThreads;
        if (i < npairs) pairs[i] = v[u];
      }
    }
  }
  __syncthreads();
  // Pair (h, seg) with k = h / heads and hh = h % heads worked out once a head.
  auto pair = [&](int k, int hh, int seg) {
    return staged ? pairs[(k * nseg + seg) * heads + hh] : __ldcg(slot(k, seg) + hh);
  };
  if (staged && nseg <= kQkNormFastSeg && Hq <= kQkNormThreads) {
    // Few segments (the usual case): thread h < Hq merges head h's pairs from
    // shared memory in segment order; no shuffles.
    if (tid < Hq) {
      const int k = tid / heads, hh = tid - k * heads;
      const float2* v = pairs + (size_t)k * per_k + hh;
      float M = -INFINITY, S = 0.0f;
#pragma unroll 8
      for (int i = 0; i < nseg; ++i) M = fmaxf(M, v[i * heads].x);
#pragma unroll 8
      for (int i = 0; i < nseg; ++i) {
        const float2 w = v[i * heads];
        if (w.x != -INFINITY) S += w.y * __expf(w.x - M);
      }
      ms[tid] = make_float2(M, __frcp_rn(S));
    }
  } else {
    int tph = 1;
    while (tph < 32 && 2 * tph * Hq <= kQkNormThreads) tph *= 2;
    const int part = tid & (tph - 1);
    // The loop's trip count is the same for every thread, so whole warps take
    // the shuffles; threads past Hq carry (-inf, 0).
    for (int hb = 0; hb < Hq; hb += kQkNormThreads / tph) {
      const int h = hb + tid / tph;
      const bool valid = h < Hq;
      const int k = h / heads, hh = h - k * heads;
      float M = -INFINITY;
      if (valid)
        for (int i = part; i < nseg; i += tph) M = fmaxf(M, pair(k, hh, i).x);
      for (int o = tph >> 1; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      float S = 0.0f;
      if (valid)
        for (int i = part; i < nseg; i += tph) {
          const float2 v = pair(k, hh, i);
          if (v.x != -INFINITY) S += v.y * __expf(v.x - M);
        }
      for (int o = tph >> 1; o > 0; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
      if (valid && part == 0) ms[h] = make_float2(M, __frcp_rn(S));
    }
  }
  __syncthreads();
  // exp(s - M) / S. The fast exponential's relative error (a few 1e-7 plus
  // |s - M| x 6e-8) stays far inside the step's 1e-4 relative tolerance.
  auto prob = [](float s, float2 w) { return __expf(s - w.x) * w.y; };
  auto put = [&](float* dst, const Vec& v, const float2* w) {
    if constexpr (VEC == 4)
      *reinterpret_cast<float4*>(dst) =
          make_float4(prob(v.x, w[0]), prob(v.y, w[1]), prob(v.z, w[2]), prob(v.w, w[3]));
    else
      *dst = prob(v, w[0]);
  };
  if (by_col) {
    float2 w[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) w[e] = active ? ms[my_col * VEC + e] : make_float2(0.f, 0.f);
    for (int r0 = 0; r0 < rows; r0 += rpb) {
      Vec y[kLoads];
      const bool more = r0 + rpb < rows;
      if (more) load(y, r0 + rpb);
#pragma unroll
      for (int u = 0; u < kLoads; ++u) {
        const int r = r0 + u * rpp + my_row;
        if (active && r < rows) put(row0 + (size_t)r * Hq + my_col * VEC, x[u], w);
      }
      if (more) {
#pragma unroll
        for (int u = 0; u < kLoads; ++u) x[u] = y[u];
      }
    }
  } else {
    for (int base = 0; base < n; base += kChunk) {
      Vec y[kLoads];
      const bool more = base + kChunk < n;
      if (more) load(y, base + kChunk);
#pragma unroll
      for (int u = 0; u < kLoads; ++u) {
        const int i = base + (tid + u * kQkNormThreads) * VEC;
        if (i < n) {
          float2 w[VEC];
#pragma unroll
          for (int e = 0; e < VEC; ++e) w[e] = ms[(i + e) % Hq];
          put(row0 + i, x[u], w);
        }
      }
      if (more) {
#pragma unroll
        for (int u = 0; u < kLoads; ++u) x[u] = y[u];
      }
    }
  }
}

// CTA (b, block of rows): the (max, sum) of every head of b from the splits
// of its tiles (pairs [tile = hg * B + b][split][heads]), then exp(s - M) / S
// over the block's rows.
__global__ void __launch_bounds__(kQkNormThreads)
gqa_qk_normalize_kernel(const __grid_constant__ QkNormParams p) {
  const int b = blockIdx.x / p.ctas_per_b;
  const int blk = blockIdx.x - b * p.ctas_per_b;
  const int L = clamped_len(p.seq_lens, b, p.Cmax);
  const int nsplit_b = L > 0 ? (L + p.rows_per_split - 1) / p.rows_per_split : 1;
  // A block past the length has nothing to do (and nothing to wait for).
  const int c0 = blk * p.rows_per_cta;
  const int c1 = min(c0 + p.rows_per_cta, L);
  if (c0 >= c1) return;
  __shared__ float2 ms[kQkMaxHeads * 32];  // (M, 1 / S) per head, Hq <= 2048
  __shared__ float2 pairs[kQkNormMaxPairs];
  auto slot = [&](int hg, int s) {
    return p.stats + ((size_t)(hg * p.B + b) * p.nsplit + s) * p.heads;
  };
  float* attn_b = p.attn + (size_t)b * p.Cmax * p.Hq;
  if (qk_norm_vec(p.Hq) == 4)
    qk_normalize_rows<4>(attn_b, p.Hq, p.heads, nsplit_b, c0, c1, slot, ms, pairs);
  else
    qk_normalize_rows<1>(attn_b, p.Hq, p.heads, nsplit_b, c0, c1, slot, ms, pairs);
}

}  // namespace gqa_av
