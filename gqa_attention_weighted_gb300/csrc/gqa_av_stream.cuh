// GQA AV decode reduction on the tcgen05 tensor cores, streamed: one
// persistent CTA per SM (or two) takes an equal share of the whole call's
// pipeline stages, across tile and sequence boundaries, through one ring.
//
// Operation (page "pytorch/executorch pull 21063", summary paragraph):
//   out[b, q_h, d] = sum_{c < L_b} attn[b, c, q_h] * V[b, c, q_h / G, d],
// with each V row read from HBM once for all heads of its group (the
// GQA-reuse paragraph on the same page).
//
// Schedule. Sequence b has n_b = max(1, ceil(L_b / R)) stages of R context
// rows (an empty sequence keeps one stage of zero weight, so its output is
// written as zeros) in each of its K = hgroups * ndt tiles (head group,
// column tile). Tile column k lists the stages of tile k of every sequence,
// sequence after sequence: T = sum_b n_b stages, the same for every column.
// The grid is U = K * Ug CTAs; CTA u takes column k = u % K and, with
// Ug' = min(Ug, T), stages [floor(T g / Ug'), floor(T (g + 1) / Ug')) of it,
// g = u / K (none when g >= Ug'). Every CTA that streams thus has the same
// number of stages (to one) whatever the lengths, there are no waves, and the
// K CTAs of a group read the same context rows of all KV heads and column
// tiles at about the same time, so each V row's bytes are fetched from DRAM
// together. A CTA's range cuts at most two tiles, the first and the last it
// touches. Each run of one tile's stages inside a CTA is a segment; a segment
// that covers its whole tile writes `out`, a cut one writes its partial to
// workspace slot 2u (the CTA's first segment) or 2u + 1 (its last), and
// gqa_av_combine_kernel<kCombineStream> adds a tile's partials in group
// order, so the result is bitwise reproducible.
//
// Per stage the arithmetic is the tensor-core kernel's (gqa_av_mma.cuh):
//   D[m][n] = sum_k V[c0 + k][d0 + m] * w[c0 + k][n]
// with V^T read in place from the 128-byte-swizzled TMA stage (A, MN-major),
// the fp32 weights split into 16-bit hi and lo rows of V's type (B,
// K-major), D double-buffered in tensor memory, and the accumulator warps
// adding hi + lo into fp32 registers stage by stage; at the end of a segment
// they store it and start the next segment from zero while the pipeline keeps
// streaming.
//
// Warp roles as in the tensor-core kernel: 4 accumulator warps, 2 or 4
// converter warps, one TMA producer warp, one warp that owns tensor memory
// and one of whose threads issues the MMAs. The producer reads every length
// once after the dependency wait, works out the CTA's range and hands the
// lengths and the range to the other warps through shared memory; every
// role then walks the same stages with its own cursor. Every mbarrier wait is
// bounded; on expiry the CTA sets the device status word, lets its copies and
// MMAs in flight finish, frees its tensor memory and returns.
#pragma once

#include "gqa_av_mma.cuh"

namespace gqa_av {

constexpr int kStreamMaxB = 2048;  // lengths kept in shared memory

// The stage list position of one role: sequence b (n stages a tile) and
// stage j of the CTA's tile of it.
struct StreamCursor {
  int b, j, n;
};

__device__ __forceinline__ void stream_advance(StreamCursor& c, int B, int R, const int* lens) {
  if (++c.j < c.n) return;
  c.j = 0;
  ++c.b;
  c.n = c.b < B ? stream_stages(lens[c.b], R) : 1;
}

// The CTA's range in its column: stage count and the cursor at its first stage.
struct StreamRange {
  int count;
  int b, j;
};

// Sequence b and stage j holding stage s0 of a column: P_b <= s0 < P_b + n_b,
// P_b the stages of the sequences before b, found by a warp prefix scan in
// the integer type I. Warp-collective.
template <typename I>
__device__ __forceinline__ bool stream_locate(const int* lens, int B, int R, I s0, StreamRange& r) {
  const int lane = threadIdx.x & 31;
  I base = 0;  // P of the first sequence of this chunk of 32
  for (int b0 = 0; b0 < B; b0 += 32) {
    const int b = b0 + lane;
    const I n = b < B ? static_cast<I>(stream_stages(lens[b], R)) : I(0);
    I incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const I t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, n > 0 && s0 >= base + incl - n && s0 < base + incl);
    if (hit) {
      const int src = __ffs(hit) - 1;
      r.b = b0 + src;
      r.j = static_cast<int>(s0 - base - __shfl_sync(0xffffffffu, incl - n, src));
      return true;
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
  return false;  // unreachable: s0 < T
}

// Warp-collective (the producer warp): stores the clamped lengths in `lens`
// and works out the range of group g of Ug in a column.
__device__ __forceinline__ StreamRange stream_range(const int32_t* seq_lens, int B, int Cmax,
                                                    int R, int g, int Ug, int* lens) {
  const int lane = threadIdx.x & 31;
  long long T = 0;
  for (int b = lane; b < B; b += 32) {
    const int L = clamped_len_ro(seq_lens, b, Cmax);
    lens[b] = L;
    T += stream_stages(L, R);
  }
  __syncwarp();  // the warp's lanes read each other's lengths below
  if (__all_sync(0xffffffffu, T < (1LL << 26))) {
    // 32 partial sums below 2^26 add up to less than 2^31: one warp reduction.
    T = __reduce_add_sync(0xffffffffu, static_cast<unsigned>(T));
  } else {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) T += __shfl_xor_sync(0xffffffffu, T, o);
  }
  StreamRange r;
  r.b = 0; r.j = 0; r.count = 0;
  // With fewer stages than groups only the first T groups take one each:
  // every CTA that streams has at least one stage (the combine relies on it).
  if (static_cast<long long>(Ug) > T) Ug = static_cast<int>(T);
  if (g >= Ug) return r;
  bool found;
  if (T < (1LL << 31) && Ug < (1 << 15)) {
    // The usual sizes, in 32-bit arithmetic: with T = q Ug + r0,
    // floor(T g / Ug) = q g + floor(r0 g / Ug), and r0 g < 2^30.
    const unsigned t = static_cast<unsigned>(T), ug = static_cast<unsigned>(Ug);
    const unsigned q = t / ug, r0 = t - q * ug;
    const unsigned s0 = q * g + (r0 * g) / ug;
    const unsigned s1 = q * (g + 1) + (r0 * (g + 1)) / ug;
    r.count = static_cast<int>(s1 - s0);
    found = stream_locate<int>(lens, B, R, static_cast<int>(s0), r);
  } else {
    const long long s0 = stream_first(T, g, Ug);
    r.count = static_cast<int>(stream_first(T, g + 1, Ug) - s0);
    found = stream_locate<long long>(lens, B, R, s0, r);
  }
  if (!found) r.count = 0;  // unreachable: s0 < T
  return r;
}

// Shared memory (offsets from a 1024-byte-aligned base): the tensor-core
// kernel's layout (V ring, attn ring, B ring, mbarriers, tensor-memory
// address, a 16-int range record) followed by the lengths at lens_off.
template <typename Tag, int NB>
__global__ void __launch_bounds__(kMmaMaxThreads, NB == 1 ? 3 : (NB == 2 ? 2 : 1))
    gqa_av_stream_kernel(const __grid_constant__ Params p) {
  constexpr int N = 16 * NB;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_addr(smem_raw);
  const uint32_t base_s = (raw_s + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base_s - raw_s);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int cvt_warps = p.cvt_warps;
  const int producer_warp = kMmaAccWarps + cvt_warps;
  const int issuer_warp = producer_warp + 1;
  const int K = p.hgroups * p.ndt;
  const int u = blockIdx.x;
  const int k = u % K;                      // the CTA's tile column
  const int hg = k / p.ndt, dti = k - (k / p.ndt) * p.ndt;
  const int h0 = hg * p.heads, kv_h = h0 / p.G, d0 = dti * p.dt;

  const uint32_t vring_s = base_s;
  const uint32_t aring_s = base_s + p.a_off;
  const uint32_t bring_s = base_s + p.b_off;
  float* aring = reinterpret_cast<float*>(smem + p.a_off);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.bar_off);
  const uint32_t full0 = smem_addr(bars);
  const uint32_t empty0 = smem_addr(bars + kMaxStages);
  const uint32_t bready0 = smem_addr(bars + 2 * kMaxStages);
  const uint32_t dfull0 = smem_addr(bars + 3 * kMaxStages);
  const uint32_t dfree0 = smem_addr(bars + 3 * kMaxStages + 2);
  const uint32_t drain = smem_addr(bars + 3 * kMaxStages + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * kMaxStages + 5);
  int* range_rec = reinterpret_cast<int*>(bars + 3 * kMaxStages + 6);
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
      mbar_init(full0 + 8 * s, p.attn_tma ? 1 : 1 + 32);
      mbar_init(empty0 + 8 * s, 1);           // one tcgen05.commit per stage
      mbar_init(bready0 + 8 * s, cvt_warps);  // one arrival per converter warp
    }
    for (int j = 0; j < 2; ++j) {
      mbar_init(dfull0 + 8 * j, 1);
      mbar_init(dfree0 + 8 * j, kMmaAccWarps);
    }
    mbar_init(drain, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == producer_warp && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.v_map)) : "memory");
    if (p.attn_tma)
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.a_map)) : "memory");
  }
  const uint64_t policy = evict_first_policy();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  grid_dependency_wait();
  grid_launch_dependents();

  // The CTA's range, worked out by the producer warp and handed over at
  // named barrier 3 with the lengths.
  StreamRange rg;
  if (warp == producer_warp) {
    rg = stream_range(p.seq_lens, p.B, p.Cmax, p.R, u / K, p.split_units / K, lens);
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
  StreamCursor cur{rg.b, rg.j, n_iters > 0 ? stream_stages(lens[rg.b], p.R) : 1};

  if (warp == producer_warp) {
    // ----------------------------------------------------------------- producer
    const int per_row = p.avec == 4 ? p.heads >> 2 : (p.avec == 2 ? p.heads >> 1 : p.heads);
    bool ok = true;
    int issued = 0;
    int stage = 0;
    uint32_t parity = 1;  // of the empty barrier: a fresh slot passes at once
    for (int it = 0; it < n_iters; ++it) {
      if (it >= p.stages && !mbar_wait(empty0 + 8 * stage, parity, p.timeout_ns)) {
        atomicOr(p.status, kErrEmptyWait);
        ok = false;
        break;
      }
      const int c0 = cur.j * p.R, b = cur.b;
      const uint32_t full = full0 + 8 * stage;
      if (lane == 0) {
        mbar_arrive_expect_tx(full, (uint32_t)p.v_halves * (p.v_stage_bytes / 2) +
                                        (p.attn_tma ? p.a_stage_bytes : 0u));
        const uint32_t vdst = vring_s + (uint32_t)stage * p.v_stage_bytes;
        for (int h = 0; h < p.v_halves; ++h)
          tma_load_4d(vdst + (uint32_t)h * p.v_stage_bytes / 2, &p.v_map, d0 + 64 * h, kv_h, c0, b,
                      full, policy);
        if (p.attn_tma)
          tma_load_3d(aring_s + (uint32_t)stage * p.a_stage_bytes, &p.a_map, h0 - (h0 & 3), c0, b,
                      full, policy);
      }
      if (!p.attn_tma) {
        // Unaligned head groups: the weights of the stage's in-range rows by cp.async.
        const int rows = max(0, min(p.R, lens[b] - c0));
        const float* src = p.attn + ((size_t)b * p.Cmax + c0) * p.Hq + h0;
        const uint32_t dst = aring_s + 4u * (uint32_t)(stage * p.R * p.ap);
        const int n = rows * per_row;
        for (int i = lane; i < n; i += 32) {
          const int r = i / per_row, col = (i - r * per_row) * p.avec;
          const uint32_t d = dst + 4u * (r * p.ap + col);
          const float* sp = src + (size_t)r * p.Hq + col;
          if (p.avec == 4) cp_async<16>(d, sp);
          else if (p.avec == 2) cp_async<8>(d, sp);
          else cp_async<4>(d, sp);
        }
        cp_async_arrive_noinc(full);
      }
      issued = it + 1;
      stream_advance(cur, p.B, p.R, lens);
      if (++stage == p.stages) { stage = 0; parity ^= 1u; }
    }
    cp_async_wait_all();
    if (!ok) {
      for (int it = max(0, issued - p.stages); it < issued; ++it)
        if (!mbar_wait(full0 + 8 * (it % p.stages), (it / p.stages) & 1, p.timeout_ns))
          atomicOr(p.status, kErrDrain);
    }
    return;
  }

  const uint32_t b_half = (uint32_t)N * p.R * 2;  // bytes of one of hi / lo

  if (warp == issuer_warp) {
    // -------------------------------------------------------------- MMA issuer
    const uint32_t idesc = mma_idesc<Tag>(2 * N);
    const uint32_t a_lbo = (uint32_t)p.R * 128;        // second 64-column half
    const uint32_t b_sbo = (uint32_t)(p.R / 8) * 128;  // next 8 rows of B
    if (lane == 0) {
      int issued = 0;
      int stage = 0;
      uint32_t phase = 0;
      for (int it = 0; it < n_iters; ++it) {
        const int j = it & 1;
        if (!mbar_poll(bready0 + 8 * stage, phase, p.timeout_ns) ||
            (it >= 2 && !mbar_poll(dfree0 + 8 * j, ((it - 2) >> 1) & 1, p.timeout_ns))) {
          atomicOr(p.status, kErrMmaWait);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(j * 2 * N);
        const uint32_t a0 = vring_s + (uint32_t)stage * p.v_stage_bytes;
        const uint32_t bb = bring_s + (uint32_t)stage * 2 * b_half;
        const uint64_t ad0 = smem_desc(a0, a_lbo, 1024, 2);
        const uint64_t bd0 = smem_desc(bb, 128, b_sbo, 0);
        mma_f16(d_tmem, ad0, bd0, idesc, 0u);
#pragma unroll 4
        for (int kk = 1; kk < p.R / 16; ++kk)
          mma_f16(d_tmem, ad0 + (uint64_t)(kk * (2048 >> 4)), bd0 + (uint64_t)(kk * (256 >> 4)),
                  idesc, 1u);
        mma_commit(empty0 + 8 * stage);  // V, attn and B slots free once these MMAs are done
        mma_commit(dfull0 + 8 * j);
        issued = it + 1;
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

  if (warp >= kMmaAccWarps) {
    // --------------------------------------------------------------- converters
    // Weights of each stage -> B hi / lo (K-major 8 x 16 B core matrices):
    // element (n, k) at ((n / 8) * nkc + k / 8) * 128 + (n % 8) * 16 + (k % 8) * 2.
    const int ctid = tid - 32 * kMmaAccWarps;
    const int nkc = p.R / 8;
    const int items = N * nkc;
    int stage = 0;
    uint32_t phase = 0;
    for (int it = 0; it < n_iters; ++it) {
      if (!mbar_poll(full0 + 8 * stage, phase, p.timeout_ns)) {
        atomicOr(p.status, kErrFullWait);
        break;
      }
      const int valid = max(0, min(p.R, lens[cur.b] - cur.j * p.R));
      const float* ast = aring + (size_t)stage * p.R * p.ap + (p.attn_tma ? (h0 & 3) : 0);
      uint8_t* bst = smem + p.b_off + (size_t)stage * 2 * b_half;
      for (int t = ctid; t < items; t += cvt_warps * 32) {
        const int n = t % N, kc = t / N;
        float w[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int k = kc * 8 + e;
          w[e] = (n < p.heads && k < valid) ? ast[(size_t)k * p.ap + n] : 0.0f;
        }
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) split_weights(Tag{}, w[2 * q], w[2 * q + 1], hi[q], lo[q]);
        const size_t off = (size_t)((n >> 3) * nkc + kc) * 128 + (n & 7) * 16;
        *reinterpret_cast<uint4*>(bst + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(bst + b_half + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
      // V rows past the context: zero (they may hold anything, NaN included).
      if (valid < p.R) {
        uint8_t* vst = smem + (size_t)stage * p.v_stage_bytes;
        const int chunks = (p.R - valid) * 8;  // 16-byte chunks of one half
        for (int t = ctid; t < chunks * p.v_halves; t += cvt_warps * 32) {
          const int h = t / chunks, c = t - h * chunks;
          const int k = valid + c / 8;
          const size_t off = (size_t)h * (p.v_stage_bytes / 2) + (size_t)(k >> 3) * 1024 +
                             (size_t)(k & 7) * 128 + (size_t)(c & 7) * 16;
          *reinterpret_cast<uint4*>(vst + off) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(bready0 + 8 * stage);
      stream_advance(cur, p.B, p.R, lens);
      if (++stage == p.stages) { stage = 0; phase ^= 1u; }
    }
    return;
  }

  // -------------------------------------------------------------- accumulators
  // Thread t owns output column m = t (tensor-memory lane t) of every head.
  const int m = tid;
  const float unscale = weight_unscale(Tag{});
  const int tile_elems = p.heads * p.dt;
  float acc[N];
#pragma unroll
  for (int n = 0; n < N; ++n) acc[n] = 0.0f;
  bool first_segment = true;
  int seg_j0 = rg.j;  // stage of the tile the current segment started at
  for (int it = 0; it < n_iters; ++it) {
    const int j = it & 1;
    if (!mbar_wait(dfull0 + 8 * j, (it >> 1) & 1, p.timeout_ns)) {
      atomicOr(p.status, kErrMmaWait);
      break;
    }
    tc_fence_after();
    const uint32_t taddr = tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)(j * 2 * N);
#pragma unroll
    for (int q = 0; q < NB; ++q) {
      float h[16], l[16];
      tmem_ld16(taddr + 16u * q, h);
      tmem_ld16(taddr + (uint32_t)N + 16u * q, l);
#pragma unroll
      for (int i = 0; i < 16; ++i) acc[16 * q + i] += h[i] + l[i];
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(dfree0 + 8 * j);
    const bool tile_end = cur.j == cur.n - 1;
    if (tile_end || it == n_iters - 1) {
      // End of a segment: the whole tile goes to out, a cut one to its slot.
      const bool whole = seg_j0 == 0 && tile_end;
      float* part = p.ws + (size_t)(2 * u + (first_segment ? 0 : 1)) * tile_elems;
      if (m < p.dt && d0 + m < p.D) {
#pragma unroll
        for (int n = 0; n < N; ++n) {
          if (n < p.heads) {
            const float v = acc[n] * unscale;
            if (whole) p.out[((size_t)cur.b * p.Hq + h0 + n) * p.D + d0 + m] = v;
            else __stcg(part + (size_t)n * p.dt + m, v);
          }
        }
      }
#pragma unroll
      for (int n = 0; n < N; ++n) acc[n] = 0.0f;
      first_segment = false;
      seg_j0 = 0;
    }
    stream_advance(cur, p.B, p.R, lens);
  }
  tc_fence_before();
  mma_team_sync();
}

// Launch and occupancy of one instantiation (defined with the instantiations).
template <typename Tag, int NB>
cudaError_t launch_stream(const Params& p, int grid, int smem_bytes, cudaStream_t stream);
template <typename Tag, int NB>
cudaError_t occupancy_stream(int smem_limit, int smem_bytes, int* ctas_per_sm);

}  // namespace gqa_av
