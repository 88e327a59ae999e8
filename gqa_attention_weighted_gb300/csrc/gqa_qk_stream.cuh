// Decode score step on the tcgen05 tensor cores, streamed: persistent CTAs
// take equal runs of the call's 128-row stages, sequence after sequence, in
// the AV reduction's streamed schedule (gqa_av_stream.cuh).
//
// Operation (the step before the AV coop-GEMV of page "pytorch/executorch
// pull 21063", summary paragraph; include/gqa_qk.h):
//   s[b, c, q_h]    = scale * sum_d q[b, q_h, d] * K[b, c, q_h / G, d],
//   attn[b, c, q_h] = exp(s - M) / S over c < L_b,
// with each K row read from HBM once for the G query heads of its group.
//
// Schedule. Sequence b has n_b = max(1, ceil(L_b / 128)) stages in each of
// its K = hgroups tiles (one head group each); tile column k lists tile k of
// every sequence, sequence after sequence, T = sum_b n_b stages. The grid is
// U = K * Ug CTAs; CTA u takes column k = u % K and, with Ug' = min(Ug, T),
// stages [floor(T g / Ug'), floor(T (g + 1) / Ug')) of it, g = u / K. The K
// CTAs of a group read the same context rows of every KV head at about the
// same time. A run of one tile's stages inside a CTA is a segment; at its
// end the CTA writes the segment's (max, sum of exp) per head: for a segment
// that is its whole tile to the tile's own slot, for a cut one to slot 2u
// (the CTA's first segment) or 2u + 1 (its last). gqa_qk_stream_normalize
// merges a tile's pairs in a fixed order and rewrites the scores, so the
// result is bitwise reproducible.
//
// Per stage of 128 context rows the CTA computes
//   S[m][n] = sum_k K[c0 + m][k] * Q[n][k]
// as D/16 `tcgen05.mma.cta_group::1.kind::f16` instructions (M = 128 rows,
// N = 2 * Npad, K = D) accumulating in fp32 in tensor memory:
//   * A = the K rows in place from the TMA stage (K-major, 128-byte swizzle,
//     D/64 parts of 128 rows x 128 B);
//   * B = the group's queries of the segment's sequence, split once per
//     segment into hi = round16(q) and lo = round16(q - hi) of K's type (hi
//     rows then lo rows, K-major core matrices), double-buffered by segment;
//   * D double-buffered in tensor memory; the four accumulator warps (one
//     context row a thread) add hi + lo, scale, write the row's scores and
//     keep a running (max, sum of exp) per head.
//
// Warps: 0-3 accumulate, 4 converts each segment's queries (with at most 16
// heads, warps 0-4 convert the first segment's together), 5 is the TMA
// producer, 6 owns tensor memory and one of its threads issues the MMAs.
// Every mbarrier wait is bounded; on expiry the CTA sets the device status
// word, lets its copies and MMAs in flight finish, frees its tensor memory and
// returns.
#pragma once

#include "gqa_av_stream.cuh"
#include "gqa_qk_mma.cuh"

namespace gqa_av {

constexpr int kQkStreamWarps = kMmaAccWarps + 3;  // + converter, producer, MMA warps
constexpr int kQkStreamThreads = 32 * kQkStreamWarps;

// Shared memory (offsets from a 1024-byte-aligned base):
//   [K ring: stages x D/64 parts x 128 rows x 128 B]             (stage_bytes each)
//   [B: 2 buffers x (hi, lo) x Npad rows x D columns, 16-bit]    at b_off
//   [reduction: 4 warps x Npad float2]                            at red_off
//   [mbarriers: full, empty (kMaxStages each), dfull[2], dfree[2], qready[2],
//    qfree[2], drain] [tensor-memory address] [range record]      at bar_off
//   [lengths: B ints]                                             at lens_off
template <typename Tag, int NB>
__global__ void __launch_bounds__(kQkStreamThreads, 1)
    gqa_qk_stream_kernel(const __grid_constant__ QkParams p) {
  constexpr int N = 16 * NB;  // Npad
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_addr(smem_raw);
  const uint32_t base_s = (raw_s + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base_s - raw_s);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  constexpr int cvt_warp = kMmaAccWarps;
  constexpr int producer_warp = kMmaAccWarps + 1;
  constexpr int issuer_warp = kMmaAccWarps + 2;
  const int K = p.hgroups;
  const int u = blockIdx.x;
  const int hg = u % K;                      // the CTA's tile column: head group hg
  const int h0 = hg * p.heads, kv_h = h0 / p.G;

  float2* red = reinterpret_cast<float2*>(smem + p.red_off);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.bar_off);
  const uint32_t full0 = smem_addr(bars);
  const uint32_t empty0 = smem_addr(bars + kMaxStages);
  const uint32_t dfull0 = smem_addr(bars + 2 * kMaxStages);
  const uint32_t dfree0 = smem_addr(bars + 2 * kMaxStages + 2);
  const uint32_t qready0 = smem_addr(bars + 2 * kMaxStages + 4);
  const uint32_t qfree0 = smem_addr(bars + 2 * kMaxStages + 6);
  const uint32_t drain = smem_addr(bars + 2 * kMaxStages + 8);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kMaxStages + 9);
  int* range_rec = reinterpret_cast<int*>(bars + 2 * kMaxStages + 10);  // 8 ints, 0-4 used
  // The first segment's queries, converted by the accumulator and converter
  // warps together (N = 16): in the range record's last 8 bytes.
  const uint32_t q0ready = smem_addr(bars + 2 * kMaxStages + 13);
  constexpr bool kFirstTogether = N == 16;
  constexpr int kFirstWarps = kMmaAccWarps + 1;
  int* lens = reinterpret_cast<int*>(smem + p.lens_off);

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
      mbar_init(qready0 + 8 * j, 1);  // the converter warp's arrival
      mbar_init(qfree0 + 8 * j, 1);   // a tcgen05.commit after a segment's last MMA
    }
    mbar_init(drain, 1);
    mbar_init(q0ready, kFirstWarps);  // one arrival per converting warp
    range_rec[4] = 0;  // the accumulators' abort flag
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

  // The CTA's range in its column, worked out by the producer warp and
  // handed over at named barrier 3 with the lengths.
  StreamRange rg;
  if (warp == producer_warp) {
    rg = stream_range(p.seq_lens, p.B, p.Cmax, kQkMmaRows, u / K, p.split_units / K, lens);
    if (lane == 0) {
      range_rec[0] = rg.count;
      range_rec[1] = rg.b;
      range_rec[2] = rg.j;
    }
    named_arrive(3, blockDim.x);
  } else {
    named_sync(3, blockDim.x);
    rg.count = range_rec[0];
    rg.b = range_rec[1];
    rg.j = range_rec[2];
  }
  const int n_iters = rg.count;
  StreamCursor cur{rg.b, rg.j, n_iters > 0 ? stream_stages(lens[rg.b], kQkMmaRows) : 1};

  const int nkc = p.D / 8;                        // 16-byte core-matrix columns along K
  const uint32_t b_half = (uint32_t)N * p.D * 2;  // bytes of the hi (or lo) rows of one buffer

  // With at most 16 heads (N = 16, at most 16 x 32 items) the first
  // segment's queries are converted into buffer 0 by the four accumulator
  // warps and the converter warp together, in one round of loads: one warp
  // alone needed two rounds, and on an MQA-shaped call the first MMA waited
  // about 4 us for them.
  if (kFirstTogether && n_iters > 0 && warp < kFirstWarps) {
    float4 x[4][2];
    const float* q_rows = p.q + ((size_t)rg.b * p.Hq + h0) * p.D;
    load_queries<N, 4>(q_rows, p.heads, nkc, tid, 32 * kFirstWarps, x);
    store_queries<Tag, N, 4>(x, nkc, smem + p.b_off, b_half, tid, 32 * kFirstWarps);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) mbar_arrive(q0ready);
  }

  if (warp == producer_warp) {
    // ----------------------------------------------------------------- producer
    bool ok = true;
    int issued = 0;
    int stage = 0;
    uint32_t parity = 1;  // of the empty barrier: a fresh slot passes at once
    for (int it = 0; it < n_iters; ++it) {
      if (it >= p.stages && !mbar_poll(empty0 + 8 * stage, parity, p.timeout_ns)) {
        if (lane == 0) atomicOr(p.status, kErrEmptyWait);
        ok = false;
        break;
      }
      if (lane == 0) {
        const uint32_t full = full0 + 8 * stage;
        mbar_arrive_expect_tx(full, p.stage_bytes);
        const uint32_t dst = base_s + (uint32_t)stage * p.stage_bytes;
        for (int part = 0; part < p.parts; ++part)
          tma_load_4d(dst + (uint32_t)part * kQkMmaRows * 128, &p.k_map, 64 * part, kv_h,
                      cur.j * kQkMmaRows, cur.b, full, policy);
      }
      issued = it + 1;
      stream_advance(cur, p.B, kQkMmaRows, lens);
      if (++stage == p.stages) { stage = 0; parity ^= 1u; }
    }
    if (!ok) {
      for (int it = max(0, issued - p.stages); it < issued; ++it)
        if (!mbar_wait(full0 + 8 * (it % p.stages), (it / p.stages) & 1, p.timeout_ns) && lane == 0)
          atomicOr(p.status, kErrDrain);
    }
    return;
  }

  if (warp == cvt_warp) {
    // ------------------------------------------------------- query converter
    // Segment e's queries -> B buffer e & 1 (element (n, k) at ((n / 8) * nkc
    // + k / 8) * 128 + (n % 8) * 16 + (k % 8) * 2; heads past the group zero).
    int e = 0;
    for (int it = 0; it < n_iters; ++it) {
      const bool seg_start = it == 0 || cur.j == 0;
      if (seg_start && kFirstTogether && e == 0) {
        ++e;  // converted above, with the accumulator warps
      } else if (seg_start) {
        const int buf = e & 1;
        if (e >= 2 && !mbar_wait(qfree0 + 8 * buf, ((e - 2) >> 1) & 1, p.timeout_ns)) {
          if (lane == 0) atomicOr(p.status, kErrMmaWait);
          break;
        }
        convert_queries<Tag, N, 8>(p.q + ((size_t)cur.b * p.Hq + h0) * p.D, p.heads, nkc,
                                   smem + p.b_off + (size_t)buf * 2 * b_half, b_half, lane, 32);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(qready0 + 8 * buf);
        ++e;
      }
      stream_advance(cur, p.B, kQkMmaRows, lens);
    }
    return;
  }

  if (warp == issuer_warp) {
    // -------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = qk_mma_idesc<Tag>(2 * N);
      int issued = 0, e = -1;
      int stage = 0;
      uint32_t phase = 0;
      for (int it = 0; it < n_iters; ++it) {
        const int j = it & 1;
        const bool seg_start = it == 0 || cur.j == 0;
        const bool seg_end = cur.j == cur.n - 1 || it == n_iters - 1;
        if (seg_start) {
          ++e;
          // Segment 0 (converted together) completes q0ready; then buffer 0's
          // qready first completes for segment 2.
          const bool first = kFirstTogether && e == 0;
          const uint32_t bar = first ? q0ready : qready0 + 8 * (e & 1);
          const uint32_t parity =
              first ? 0u : (kFirstTogether && (e & 1) == 0 ? ((e >> 1) - 1) & 1 : (e >> 1) & 1);
          if (!mbar_poll(bar, parity, p.timeout_ns)) {
            atomicOr(p.status, kErrMmaWait);
            break;
          }
        }
        if (!mbar_poll(full0 + 8 * stage, phase, p.timeout_ns) ||
            (it >= 2 && !mbar_poll(dfree0 + 8 * j, ((it - 2) >> 1) & 1, p.timeout_ns))) {
          atomicOr(p.status, kErrMmaWait);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(j * 2 * N);
        const uint32_t a0 = base_s + (uint32_t)stage * p.stage_bytes;
        const uint64_t bd0 =
            smem_desc(base_s + p.b_off + (uint32_t)(e & 1) * 2 * b_half, 128, (uint32_t)nkc * 128, 0);
        for (int kk = 0; kk < p.D / 16; ++kk) {
          // K step kk: part kk / 4 (128 x 128 B each), 32 B into it per step.
          const uint32_t a_addr =
              a0 + (uint32_t)(kk >> 2) * kQkMmaRows * 128 + (uint32_t)(kk & 3) * 32;
          mma_f16(d_tmem, smem_desc(a_addr, 16, 1024, 2), bd0 + (uint64_t)(kk * (256 >> 4)),
                  idesc, kk > 0 ? 1u : 0u);
        }
        mma_commit(empty0 + 8 * stage);  // the K slot is free once these MMAs are done
        mma_commit(dfull0 + 8 * j);
        if (seg_end) mma_commit(qfree0 + 8 * (e & 1));  // and the segment's queries
        issued = it + 1;
        stream_advance(cur, p.B, kQkMmaRows, lens);
        if (++stage == p.stages) { stage = 0; phase ^= 1u; }
      }
      if (issued > 0) {
        mma_commit(drain);
        if (!mbar_wait(drain, 0, p.timeout_ns)) atomicOr(p.status, kErrMmaWait);
      }
    }
    __syncwarp();
    mma_team_sync();  // the accumulators are done with tensor memory
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(p.tmem_cols)
                 : "memory");
    return;
  }

  // -------------------------------------------------------------- accumulators
  const int m_row = tid;  // tensor-memory lane = context row of the stage
  float mx[N], sm[N];
#pragma unroll
  for (int n = 0; n < N; ++n) {
    mx[n] = -INFINITY;
    sm[n] = 0.0f;
  }
  bool first_segment = true;
  int seg_j0 = rg.j;
  // Every accumulator warp walks every stage and reaches every named barrier
  // of the segment ends, also after a bounded wait ran out (in any of them:
  // the flag below), so no barrier waits for a warp that left.
  volatile int* abort_flag = range_rec + 4;
  bool ok = true;
  // attn rows are 16-byte aligned (checked on the host) and so is head h0 of
  // a group of a multiple of 4 heads.
  const bool vec4 = p.heads % 4 == 0 && p.Hq % 4 == 0;
  for (int it = 0; it < n_iters; ++it) {
    const int j = it & 1;
    if (ok && (*abort_flag || !mbar_poll(dfull0 + 8 * j, (it >> 1) & 1, p.timeout_ns))) {
      if (!*abort_flag) atomicOr(p.status, kErrMmaWait);
      *abort_flag = 1;
      ok = false;
    }
    ok = __all_sync(0xffffffffu, ok);
    float s[N];
    if (ok) {
      tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)(j * 2 * N);
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
    }
    const int L = lens[cur.b];
    const int c = cur.j * kQkMmaRows + m_row;
    if (ok && c < L) {
      float* dst = p.attn + ((size_t)cur.b * p.Cmax + c) * p.Hq + h0;
      // The row's scores as 16-byte stores where the group's heads allow it
      // (whole 32-byte sectors, not scattered 4-byte pieces), else one by one.
      if (vec4) {
#pragma unroll
        for (int n = 0; n < N; n += 4)
          if (n < p.heads)
            __stcg(reinterpret_cast<float4*>(dst + n), make_float4(s[n], s[n + 1], s[n + 2], s[n + 3]));
      }
      if (!vec4) {
#pragma unroll
        for (int n = 0; n < N; ++n)
          if (n < p.heads) dst[n] = s[n];
      }
      online_lse_update<N>(mx, sm, s, p.heads);
    }
    const bool tile_end = cur.j == cur.n - 1;
    if (tile_end || it == n_iters - 1) {
      // End of a segment: one (max, sum) per head, over each warp's lanes and
      // then over the four warps in warp order, to the tile's slot (whole) or
      // the CTA's (cut).
      warp_lse_heads<N>(mx, sm, p.heads, red + (size_t)warp * N);  // the group's heads only
#pragma unroll
      for (int n = 0; n < N; ++n) {
        mx[n] = -INFINITY;
        sm[n] = 0.0f;
      }
      named_sync(1, 32 * kMmaAccWarps);
      if (tid < p.heads) {
        const bool whole = seg_j0 == 0 && tile_end;
        float2* dst = whole ? p.stats_whole + ((size_t)cur.b * K + hg) * p.heads
                            : p.stats + (size_t)(2 * u + (first_segment ? 0 : 1)) * p.heads;
        const float2 r = lse_of(red + tid, kMmaAccWarps, N);
        if (!*abort_flag) dst[tid] = r;
      }
      named_sync(1, 32 * kMmaAccWarps);  // red is reused by the next segment
      first_segment = false;
      seg_j0 = 0;
    }
    stream_advance(cur, p.B, kQkMmaRows, lens);
  }
  tc_fence_before();
  mma_team_sync();
}

// ---------------------------------------------------------------------------
// CTA (b, block of rows): the (max, sum) of every head of b, merged over the
// segments of its tile (the tile's own slot when one CTA held it whole), then
// exp(s - M) / S over the block's rows.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kQkNormThreads)
    gqa_qk_stream_normalize(const __grid_constant__ QkNormParams p) {
  __shared__ long long span[2];            // stages of a column in all, and before b
  const int b = blockIdx.x / p.ctas_per_b;
  const int blk = blockIdx.x - b * p.ctas_per_b;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // The lengths are read before the dependency wait: the score kernel, the
  // only grid this one depends on, does not write them.
  if (warp == 0) {
    const longlong2 r = stream_prefix(p.seq_lens, p.B, p.Cmax, kQkMmaRows, b);
    if (lane == 0) {
      span[0] = r.x;
      span[1] = r.y;
    }
  }
  __syncthreads();
  const int L = clamped_len(p.seq_lens, b, p.Cmax);
  const long long T = span[0], P = span[1];
  const int nb = stream_stages(L, kQkMmaRows);
  const int K = p.hgroups;
  const int Ug0 = p.split_units / K;
  const int Ug = static_cast<int>(T < Ug0 ? T : Ug0);
  const int g0 = stream_owner(T, P, Ug), g1 = stream_owner(T, P + nb - 1, Ug);
  const int adj = stream_first(T, g0, Ug) == P ? 0 : 1;
  // A block past the length has nothing to do (and nothing to wait for).
  const int c0 = blk * p.rows_per_cta;
  const int c1 = min(c0 + p.rows_per_cta, L);
  if (c0 >= c1) return;
  // Segment i of head group k: the tile's own slot when one CTA held it
  // whole, else slot 2 (g K + k) of group g = g0 + i (2 (g0 K + k) + 1 for
  // the first when the tile does not start g0's range).
  const int nseg = g0 == g1 ? 1 : g1 - g0 + 1;
  __shared__ float2 ms[kQkMaxHeads * 32];  // (M, 1 / S) per head, Hq <= 2048
  __shared__ float2 pairs[kQkNormMaxPairs];
  auto slot = [&](int k, int i) {
    if (g0 == g1) return p.stats_whole + ((size_t)b * K + k) * p.heads;
    return p.stats + (size_t)(2 * ((g0 + i) * K + k) + (i == 0 ? adj : 0)) * p.heads;
  };
  float* attn_b = p.attn + (size_t)b * p.Cmax * p.Hq;
  if (qk_norm_vec(p.Hq) == 4)
    qk_normalize_rows<4>(attn_b, p.Hq, p.heads, nseg, c0, c1, slot, ms, pairs);
  else
    qk_normalize_rows<1>(attn_b, p.Hq, p.heads, nseg, c0, c1, slot, ms, pairs);
}

}  // namespace gqa_av
