// Fused decode attention for sm_103a (GB300): scores, softmax and the
// weighted sum of V in one pass over the KV cache, with K and V rows read
// from HBM once for all query heads of their group.
//
//   s[b, c, q_h]   = scale * sum_d q[b, q_h, d] * K[b, c, q_h / G, d]
//   out[b, q_h, :] = sum_{c < L_b} softmax_c(s)[b, c, q_h] * V[b, c, q_h / G, :]
//
// The AV coop-GEMV of LLM decode (page "pytorch/executorch pull 21063",
// summary paragraph) takes the softmax weights as an input; here the weights
// are made on chip from the same step's query-key products, so the fp32
// weight array never goes through HBM. The query-to-KV-head grouping is the
// page's GQA-reuse reading: one CTA owns the query heads of one KV head.
//
// gqa_attn_kernel: one CTA owns a tile (head chunk of one KV head, b) and a
// context split of it. A producer warp streams stages of 32 context rows of
// K and of V by 4-D TMA (64-column boxes, 128-byte swizzle) into a ring whose
// slots belong to fixed consumer warps (slot s to warp s % nw), so each warp
// waits only on its own slots. A consumer warp takes whole stages and runs an
// independent online softmax over them:
//   * scores: S[h][r] = q'[h] . K[r] with warp-level tensor-core products
//     (mma.sync m16n8k16, fp32 accumulate), M = the CTA's heads padded to 16,
//     N = 8 context rows, K = 16 columns. q' = q * scale * log2(e) is split
//     once per CTA into hi + lo halves in V's 16-bit type; K is exact in it.
//   * softmax: per head the stage maximum (a quad shuffle), the running
//     maximum m, alpha = 2^(m_old - m_new), p = 2^(S - m_new), l = l*alpha + sum p.
//   * AV: O[h][d] = O[h][d] * alpha + (P_hi + P_lo)[h][:] . V[:][d], the
//     stage's products made by the tensor core from zero and added to the
//     fp32 register accumulator with one FMA, so the tensor core never sums
//     more than one stage. P's fragments are the score fragments themselves.
// At D = 256 the output columns can be cut into two blocks of 128 owned by
// two CTAs (each computes all the scores and half of the weighted sum): a
// thread then holds 64 output sums instead of 128, and the two CTAs, adjacent
// in the grid, read the same K rows at about the same time (the second read
// is an L2 hit).
// Rows past the split or the sequence get score -inf and their V rows are
// zeroed in shared memory (they may hold NaN). At the end the warps' (m, l,
// O) are merged through shared memory in warp order; a tile whose context
// fits one split writes out = O / l, otherwise each split writes (O, m, l)
// and gqa_attn_combine_kernel, launched next with programmatic dependent
// launch, merges the splits of each (tile, head) in split order. Results are
// bitwise reproducible for a fixed launch shape.
#pragma once

#include "gqa_av_kernel.cuh"

namespace gqa_av {

constexpr int kAttnRows = 32;          // context rows per stage
constexpr int kAttnMaxWarps = 8;       // consumer warps at most
// A thread holds D / 2 fp32 output sums. Up to 6 consumer warps (7 with the
// producer, two on a sub-partition) leave it 255 registers; 8 (nine warps)
// cap it at 168. The kernel is compiled for either bound (MW = 6 or 8):
// D = 256 only for 6, D = 128 for both (8 warps spill a little but stream
// faster on many-wave grids), D = 64 for 8.
__host__ __device__ constexpr int attn_max_warps(int D) { return D == 256 ? 6 : kAttnMaxWarps; }
constexpr int kAttnMaxHeads = 16;      // query heads per CTA (one m16 tile)
constexpr int kAttnCombineThreads = 128;  // 4 columns a thread, 2 to 8 parts of the splits

struct alignas(64) AttnParams {
  CUtensorMap k_map;            // K as 4-D {D, Hkv, Cmax, B}; box {64, 1, 32, 1}, 128B swizzle
  CUtensorMap v_map;            // V, the same
  const float* q;               // [B, Hq, D]
  const int32_t* seq_lens;      // [B] or null
  float* out;                   // [B, Hq, D]
  float* ws_o;                  // [tiles][nsplit][heads][D] unnormalised split sums
  float2* ws_ml;                // [tiles][nsplit][heads] (max, sum of 2^(s - max)) per split
  unsigned int* status;         // device status word
  float qscale;                 // scale * log2(e)
  int B, Cmax, Hq, Hkv, D, G;
  int heads;                    // query heads per CTA (<= 16)
  int hgroups;                  // Hq / heads
  int ncol;                     // column blocks of the output (1, or 2 at D = 256)
  int kt;                       // tiles of one sequence: hgroups * ncol
  int nw;                       // consumer warps
  int stages;                   // ring slots, a multiple of nw
  int rows_per_split, nsplit;   // fixed splits
  int balanced;                 // splits balanced over the batch's lengths
  int units;                    // balanced: CTAs the batch's context is spread over
  uint32_t stage_bytes;         // 32 * (D + D / ncol) * 2: K rows, then the block's V columns
  uint32_t q_off;               // shared-memory offset of q' hi and lo (16 rows each)
  uint32_t qstride;             // bytes per q' row in shared memory (D * 2 + 16)
  uint32_t bar_off;             // shared-memory offset of the mbarriers and the fail flag
  long long timeout_ns;
};

struct AttnCombineParams {
  const float* ws_o;
  const float2* ws_ml;
  const int32_t* seq_lens;
  float* out;
  int B, Cmax, Hq, D, heads, hgroups, rows_per_split, nsplit;
  int balanced, units;
  int ncol, kt;                 // column blocks, tiles of one sequence
};

// ---------------------------------------------------------------------------
// Warp-level tensor-core helpers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

// d += a (16x16, row-major) * b (16x8, column-major), fp32 accumulate. Not
// volatile: a pure function of its registers, so the compiler may interleave
// independent products to hide the tensor pipe's latency.
__device__ __forceinline__ void mma16816(Bf16Tag, float (&d)[4], const uint32_t (&a)[4],
                                         uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma16816(Fp16Tag, float (&d)[4], const uint32_t (&a)[4],
                                         uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// x ~= hi + lo with hi and lo in the cache's 16-bit type; two values packed
// per register, the first in the low half.
__device__ __forceinline__ void split_pack(Bf16Tag, float x, float y, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
  const __nv_bfloat162 l =
      __floats2bfloat162_rn(x - __low2float(h), y - __high2float(h));
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

__device__ __forceinline__ void split_pack(Fp16Tag, float x, float y, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(x, y);
  const __half2 l = __floats2half2_rn(x - __low2float(h), y - __high2float(h));
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

__device__ __forceinline__ void split_one(Bf16Tag, float x, uint16_t& hi, uint16_t& lo) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  const __nv_bfloat16 l = __float2bfloat16_rn(x - __bfloat162float(h));
  hi = *reinterpret_cast<const uint16_t*>(&h);
  lo = *reinterpret_cast<const uint16_t*>(&l);
}

__device__ __forceinline__ void split_one(Fp16Tag, float x, uint16_t& hi, uint16_t& lo) {
  const __half h = __float2half_rn(x);
  const __half l = __float2half_rn(x - __half2float(h));
  hi = *reinterpret_cast<const uint16_t*>(&h);
  lo = *reinterpret_cast<const uint16_t*>(&l);
}

// fp16 weights are scaled by 2^12 before the split (exact; p <= 1 stays far
// below the fp16 maximum) so that small weights keep their bits instead of
// going subnormal; the factor is taken out before anything leaves the CTA.
__host__ __device__ constexpr float weight_gain(Bf16Tag) { return 1.0f; }
__host__ __device__ constexpr float weight_gain(Fp16Tag) { return 4096.0f; }

// 2^x for the softmax. The scores arrive multiplied by log2(e), so this is
// exp of the natural-log score; -inf gives 0.
__device__ __forceinline__ float exp2_fast(float x) { return exp2f(x); }

// ---------------------------------------------------------------------------
// Shared memory (offsets from a 1024-byte-aligned base):
//   [ring: stages x (K: D/64 parts x 32 rows x 128 B | V: the same)]
//   [q' hi: 16 x qstride][q' lo: 16 x qstride]
//   [mbarriers: full, empty (stages each)][fail flag]
// After the context loop the ring is reused for the warps' merge:
//   [O: nw x heads x (D + 4) floats][(m, l): nw x heads float2]
template <typename Tag, int D, int DV, int MW>
__global__ void __launch_bounds__(32 * (MW + 1), 1)
    gqa_attn_kernel(const __grid_constant__ AttnParams p) {
  constexpr int R = kAttnRows;
  constexpr int KS = D / 16;          // 16-column k-steps of the score product
  constexpr int NT = DV / 8;          // 8-column n-tiles of the CTA's output columns
  constexpr uint32_t kHalf = R * D * 2;  // K bytes of a stage; V follows
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_addr(smem_raw);
  const uint32_t base_s = (raw_s + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base_s - raw_s);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int nthreads = 32 * (p.nw + 1);

  // A tile is (head group hg, column block cb, b); hgv = hg * ncol + cb.
  // Fixed splits: CTA (tile, split), tile = hgv * B + b. Balanced splits: CTA
  // u takes hgv = u % kt and batch split u / kt, found from the lengths after
  // the dependency wait. Either way its partial is slot blockIdx.x.
  int hgv, b, split, c_begin, rps;
  if (!p.balanced) {
    const int tile = blockIdx.x / p.nsplit;
    split = blockIdx.x - tile * p.nsplit;
    hgv = tile / p.B;
    b = tile - hgv * p.B;
    rps = p.rows_per_split;
    c_begin = split * rps;
  } else {
    hgv = blockIdx.x % p.kt;
    b = split = c_begin = rps = 0;
  }
  const int hg = hgv / p.ncol;
  const int dv0 = (hgv - hg * p.ncol) * DV;  // first output column of the CTA
  const int h0 = hg * p.heads;
  const int kv_h = h0 / p.G;
  // Fixed splits issue their first stages before the length is read.
  const int pre =
      p.balanced ? 0 : min(min(p.stages, rps / R), (p.Cmax - c_begin + R - 1) / R);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.bar_off);
  volatile int* fail = reinterpret_cast<volatile int*>(bars + 2 * p.stages);
  const uint32_t full0 = smem_addr(bars);
  const uint32_t empty0 = smem_addr(bars + p.stages);

  if (tid == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    *fail = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == p.nw && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.k_map)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.v_map)) : "memory");
  }
  const uint64_t policy = evict_first_policy();
  __syncthreads();

  grid_dependency_wait();
  grid_launch_dependents();

  int L, nsplit_b;
  if (!p.balanced) {
    L = clamped_len(p.seq_lens, b, p.Cmax);
    nsplit_b = L > 0 ? (L + rps - 1) / rps : 1;
  } else {
    // Warp-collective: every warp works the split out for itself.
    const int sps = balanced_sps(p.seq_lens, p.B, p.Cmax, R, p.kt, p.units);
    const BalancedSplit bs = balanced_find(p.seq_lens, p.B, p.Cmax, R, sps, blockIdx.x / p.kt);
    if (bs.found) {
      b = bs.b;
      L = bs.L;
      split = bs.split;
      nsplit_b = bs.n;
    } else {  // past the batch's splits: no work
      b = 0;
      L = 0;
      split = 1;
      nsplit_b = 1;
    }
    rps = sps * R;
    c_begin = split * rps;
  }
  const int c_end = min(c_begin + rps, L);
  const int n_iters = split < nsplit_b && c_end > c_begin ? (c_end - c_begin + R - 1) / R : 0;

  if (warp == p.nw) {
    // ----------------------------------------------------------------- producer
    auto issue = [&](int stage, int c0) {
      if (lane == 0) {
        const uint32_t full = full0 + 8 * stage;
        mbar_arrive_expect_tx(full, p.stage_bytes);
        const uint32_t dst = base_s + (uint32_t)stage * p.stage_bytes;
#pragma unroll
        for (int part = 0; part < D / 64; ++part)
          tma_load_4d(dst + (uint32_t)part * R * 128, &p.k_map, 64 * part, kv_h, c0, b, full,
                      policy);
#pragma unroll
        for (int part = 0; part < DV / 64; ++part)
          tma_load_4d(dst + kHalf + (uint32_t)part * R * 128, &p.v_map, dv0 + 64 * part, kv_h, c0,
                      b, full, policy);
      }
    };
    for (int it = 0; it < pre; ++it) issue(it, c_begin + it * R);  // before the length is known
    bool ok = true;
    int issued = pre;
    for (int it = pre; it < n_iters; ++it) {
      const int stage = it % p.stages;
      if (!mbar_wait(empty0 + 8 * stage, ((it / p.stages) & 1) ^ 1, p.timeout_ns)) {
        if (lane == 0) {
          atomicOr(p.status, kErrEmptyWait);
          *fail = 1;
        }
        ok = false;
        break;
      }
      issue(stage, c_begin + it * R);
      issued = it + 1;
    }
    if (!ok) {
      for (int it = max(0, issued - p.stages); it < issued; ++it)
        if (!mbar_wait(full0 + 8 * (it % p.stages), (it / p.stages) & 1, p.timeout_ns) && lane == 0)
          atomicOr(p.status, kErrDrain);
    }
    // Early stages past the split's rows: let them land before the ring is reused.
    for (int it = n_iters; it < pre; ++it)
      if (!mbar_wait(full0 + 8 * it, 0, p.timeout_ns) && lane == 0) {
        atomicOr(p.status, kErrDrain);
        *fail = 1;
      }
  } else {
    // ---------------------------------------------------------------- consumers
    // q' = q * scale * log2(e) of the CTA's heads as 16-bit hi and lo rows;
    // rows past `heads` are zero.
    {
      // Batches of kQv float4 loads a thread, all issued before any is used.
      constexpr int kQv = 4;
      const uint32_t qs = p.qstride;
      uint8_t* qhi = smem + p.q_off;
      uint8_t* qlo = qhi + 16 * qs;
      const float4* src = reinterpret_cast<const float4*>(p.q + ((size_t)b * p.Hq + h0) * D);
      const int nthr = 32 * p.nw;
      for (int i0 = tid; i0 < 16 * D / 4; i0 += kQv * nthr) {
      float4 x[kQv];
#pragma unroll
      for (int u = 0; u < kQv; ++u) {
        const int i = i0 + u * nthr;  // float4 index: head i / (D/4), columns 4 * (i % (D/4))
        x[u] = (i < 16 * D / 4 && i / (D / 4) < p.heads) ? src[i] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kQv; ++u) {
        const int i = i0 + u * nthr;
        if (i < 16 * D / 4) {
          const int h = i / (D / 4), d = (i - h * (D / 4)) * 4;
          uint32_t hi[2], lo[2];
          split_pack(Tag{}, x[u].x * p.qscale, x[u].y * p.qscale, hi[0], lo[0]);
          split_pack(Tag{}, x[u].z * p.qscale, x[u].w * p.qscale, hi[1], lo[1]);
          *reinterpret_cast<uint2*>(qhi + h * qs + d * 2) = make_uint2(hi[0], hi[1]);
          *reinterpret_cast<uint2*>(qlo + h * qs + d * 2) = make_uint2(lo[0], lo[1]);
        }
      }
      }
    }
    named_sync(1, 32 * p.nw);

    const int g = lane >> 2;   // fragment row group: heads g and g + 8
    const int t = lane & 3;    // thread in group: columns 2t, 2t + 1
    const int mi = lane >> 3;  // ldmatrix: which 8x8 matrix this lane addresses
    const int mr = lane & 7;   // ldmatrix: which row of it
    const uint32_t qhi_s = base_s + p.q_off;
    const uint32_t qlo_s = qhi_s + 16 * p.qstride;
    // q' fragments (A operand, heads x columns): matrix mi is (heads 8*(mi&1).., chunk 2ks + (mi>>1)).
    const uint32_t q_lane = (uint32_t)(((mi & 1) * 8 + mr) * p.qstride + (mi >> 1) * 16);

    float o[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.0f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;
    const float gain = weight_gain(Tag{});

    for (int it = warp; it < n_iters; it += p.nw) {
      const int stage = it % p.stages;
      if (!mbar_wait(full0 + 8 * stage, (it / p.stages) & 1, p.timeout_ns)) {
        if (lane == 0) {
          atomicOr(p.status, kErrFullWait);
          *fail = 1;
        }
        break;
      }
      const uint32_t k_s = base_s + (uint32_t)stage * p.stage_bytes;
      const uint32_t v_s = k_s + kHalf;

      const int c0 = c_begin + it * R;
      const int nvalid = min(R, c_end - c0);

      // ---- scores S[h][r] for the stage's 32 rows (4 n-tiles of 8 rows).
      float s[4][4];
#pragma unroll
      for (int j = 0; j < 4; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.0f;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t ahi[4], alo[4];
        ldsm_x4(qhi_s + q_lane + ks * 32, ahi);
        ldsm_x4(qlo_s + q_lane + ks * 32, alo);
        const int chunk = 2 * ks + (mi & 1);
        const uint32_t part_off = (uint32_t)(chunk >> 3) * R * 128;
        const uint32_t swz = (uint32_t)(((chunk & 7) ^ mr) << 4);
        // K rows 16jp.. : matrix mi is (rows 16jp + 8*(mi>>1).., chunk 2ks + (mi&1)).
        uint32_t kb[2][4];
#pragma unroll
        for (int jp = 0; jp < 2; ++jp)
          ldsm_x4(k_s + part_off + (uint32_t)(16 * jp + 8 * (mi >> 1) + mr) * 128 + swz, kb[jp]);
        // The hi products of the four row tiles, then the lo ones: each
        // accumulator is used again only four products later.
#pragma unroll
        for (int j = 0; j < 4; ++j) mma16816(Tag{}, s[j], ahi, kb[j >> 1][2 * (j & 1)], kb[j >> 1][2 * (j & 1) + 1]);
#pragma unroll
        for (int j = 0; j < 4; ++j) mma16816(Tag{}, s[j], alo, kb[j >> 1][2 * (j & 1)], kb[j >> 1][2 * (j & 1) + 1]);
      }

      if (nvalid < R) {
        // Rows past the context: score -inf, and V zeroed in shared memory.
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int r = 8 * j + 2 * t;
          if (r >= nvalid) s[j][0] = s[j][2] = -INFINITY;
          if (r + 1 >= nvalid) s[j][1] = s[j][3] = -INFINITY;
        }
        const int lines = (R - nvalid) * (DV / 64);  // 128-byte lines to clear
        for (int i = lane; i < lines * 8; i += 32) {
          const int line = i >> 3, q16 = i & 7;
          const int r = nvalid + line / (DV / 64), part = line % (DV / 64);
          *reinterpret_cast<uint4*>(smem + (v_s - base_s) + part * R * 128 + r * 128 + q16 * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        __syncwarp();
      }

      // ---- online softmax over the stage (rows of a head lie in one quad).
      float x0 = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
      x0 = fmaxf(x0, fmaxf(fmaxf(s[2][0], s[2][1]), fmaxf(s[3][0], s[3][1])));
      float x1 = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
      x1 = fmaxf(x1, fmaxf(fmaxf(s[2][2], s[2][3]), fmaxf(s[3][2], s[3][3])));
#pragma unroll
      for (int o2 = 1; o2 <= 2; o2 <<= 1) {
        x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, o2));
        x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, o2));
      }
      const float mn0 = fmaxf(m0, x0), mn1 = fmaxf(m1, x1);
      const float ms0 = mn0 == -INFINITY ? 0.0f : mn0;  // no row yet: p = 0, alpha = 1
      const float ms1 = mn1 == -INFINITY ? 0.0f : mn1;
      const float a0 = exp2_fast(m0 - ms0);             // m0 = -inf gives 0 (O is 0 then)
      const float a1 = exp2_fast(m1 - ms1);
      m0 = mn0;
      m1 = mn1;
      float sum0 = 0.0f, sum1 = 0.0f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        s[j][0] = exp2_fast(s[j][0] - ms0);
        s[j][1] = exp2_fast(s[j][1] - ms0);
        s[j][2] = exp2_fast(s[j][2] - ms1);
        s[j][3] = exp2_fast(s[j][3] - ms1);
        sum0 += s[j][0] + s[j][1];
        sum1 += s[j][2] + s[j][3];
      }
      l0 = l0 * a0 + sum0;
      l1 = l1 * a1 + sum1;

      // ---- P as the A operand of the AV product (rows = heads, k = context rows).
      uint32_t phi[2][4], plo[2][4];
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        split_pack(Tag{}, s[2 * kk][0] * gain, s[2 * kk][1] * gain, phi[kk][0], plo[kk][0]);
        split_pack(Tag{}, s[2 * kk][2] * gain, s[2 * kk][3] * gain, phi[kk][1], plo[kk][1]);
        split_pack(Tag{}, s[2 * kk + 1][0] * gain, s[2 * kk + 1][1] * gain, phi[kk][2], plo[kk][2]);
        split_pack(Tag{}, s[2 * kk + 1][2] * gain, s[2 * kk + 1][3] * gain, phi[kk][3], plo[kk][3]);
      }

      // ---- O = O * alpha + P . V, 16 output columns (two n-tiles) at a time.
#pragma unroll
      for (int nj = 0; nj < NT / 2; ++nj) {
        // V: matrix mi is (rows 16kk + 8*(mi&1).., chunk 2nj + (mi>>1)), transposed.
        const int chunk = 2 * nj + (mi >> 1);
        const uint32_t part_off = (uint32_t)(chunk >> 3) * R * 128;
        const uint32_t swz = (uint32_t)(((chunk & 7) ^ mr) << 4);
        float d0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, d1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        uint32_t vb[2][4];
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
          ldsm_x4_trans(v_s + part_off + (uint32_t)(16 * kk + 8 * (mi & 1) + mr) * 128 + swz, vb[kk]);
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          mma16816(Tag{}, d0, phi[kk], vb[kk][0], vb[kk][1]);
          mma16816(Tag{}, d1, phi[kk], vb[kk][2], vb[kk][3]);
        }
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          mma16816(Tag{}, d0, plo[kk], vb[kk][0], vb[kk][1]);
          mma16816(Tag{}, d1, plo[kk], vb[kk][2], vb[kk][3]);
        }
        o[2 * nj][0] = fmaf(o[2 * nj][0], a0, d0[0]);
        o[2 * nj][1] = fmaf(o[2 * nj][1], a0, d0[1]);
        o[2 * nj][2] = fmaf(o[2 * nj][2], a1, d0[2]);
        o[2 * nj][3] = fmaf(o[2 * nj][3], a1, d0[3]);
        o[2 * nj + 1][0] = fmaf(o[2 * nj + 1][0], a0, d1[0]);
        o[2 * nj + 1][1] = fmaf(o[2 * nj + 1][1], a0, d1[1]);
        o[2 * nj + 1][2] = fmaf(o[2 * nj + 1][2], a1, d1[2]);
        o[2 * nj + 1][3] = fmaf(o[2 * nj + 1][3], a1, d1[3]);
      }
      if (nvalid < R) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * stage);
    }

    // l over the quad (each lane summed its own rows); m is already quad-wide.
#pragma unroll
    for (int o2 = 1; o2 <= 2; o2 <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, o2);
      l1 += __shfl_xor_sync(0xffffffffu, l1, o2);
    }
    // Wait until every warp has left the ring, then write this warp's state
    // into it (the producer joins after its early stages have landed).
    named_sync(2, nthreads);
    if (*fail) return;
    const int ostride = DV + 4;  // floats; keeps the float2 stores conflict-free
    float* mo = reinterpret_cast<float*>(smem);
    float2* mml = reinterpret_cast<float2*>(smem + (size_t)p.nw * p.heads * ostride * 4);
    const float inv_gain = 1.0f / gain;
    if (g < p.heads) {
      float* row = mo + ((size_t)warp * p.heads + g) * ostride;
#pragma unroll
      for (int n = 0; n < NT; ++n)
        *reinterpret_cast<float2*>(row + 8 * n + 2 * t) =
            make_float2(o[n][0] * inv_gain, o[n][1] * inv_gain);
      if (t == 0) mml[warp * p.heads + g] = make_float2(m0, l0);
    }
    if (g + 8 < p.heads) {
      float* row = mo + ((size_t)warp * p.heads + g + 8) * ostride;
#pragma unroll
      for (int n = 0; n < NT; ++n)
        *reinterpret_cast<float2*>(row + 8 * n + 2 * t) =
            make_float2(o[n][2] * inv_gain, o[n][3] * inv_gain);
      if (t == 0) mml[warp * p.heads + g + 8] = make_float2(m1, l1);
    }
  }
  if (warp == p.nw) {
    named_sync(2, nthreads);
    if (*fail) return;
  }
  named_sync(3, nthreads);
  if (split >= nsplit_b) return;  // a split past the sequence: nothing to write

  // ---- merge the warps in warp order, then write out or this split's partial.
  const int ostride = DV + 4;
  const float* mo = reinterpret_cast<const float*>(smem);
  const float2* mml = reinterpret_cast<const float2*>(smem + (size_t)p.nw * p.heads * ostride * 4);
  const int n4 = p.heads * (DV / 4);
  for (int i = tid; i < n4; i += nthreads) {
    const int h = i / (DV / 4), d = (i - h * (DV / 4)) * 4;
    float M = -INFINITY;
    for (int w = 0; w < p.nw; ++w) M = fmaxf(M, mml[w * p.heads + h].x);
    float l = 0.0f;
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (M != -INFINITY) {
      for (int w = 0; w < p.nw; ++w) {
        const float2 ml = mml[w * p.heads + h];
        const float e = exp2_fast(ml.x - M);  // a warp with no rows: 2^-inf = 0
        l = fmaf(ml.y, e, l);
        const float4 x = *reinterpret_cast<const float4*>(mo + ((size_t)w * p.heads + h) * ostride + d);
        acc.x = fmaf(x.x, e, acc.x);
        acc.y = fmaf(x.y, e, acc.y);
        acc.z = fmaf(x.z, e, acc.z);
        acc.w = fmaf(x.w, e, acc.w);
      }
    }
    if (nsplit_b == 1) {
      const float inv = l > 0.0f ? 1.0f / l : 0.0f;
      *reinterpret_cast<float4*>(p.out + ((size_t)b * p.Hq + h0 + h) * D + dv0 + d) =
          make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    } else {
      const size_t slot = (size_t)blockIdx.x * p.heads + h;
      __stcg(reinterpret_cast<float4*>(p.ws_o + slot * DV + d), acc);
      if (d == 0) __stcg(p.ws_ml + slot, make_float2(M, l));
    }
  }
}

// ---------------------------------------------------------------------------
// CTA per (tile, head): the splits' maxima give M and the normaliser
// Z = sum_s 2^(m_s - M) l_s; then out = sum_s 2^(m_s - M) / Z * O_s. A thread
// owns 4 output columns and the splits s = part, part + parts, ...; the
// first batch of its partial loads goes out before M and Z are known, so the
// call costs about one round trip to L2 after the dependency wait. The parts
// are added in part order, so the result is deterministic. Tiles whose
// sequence fits one split were written by the main kernel and are skipped.
// Split s of a tile is slot tile * nsplit + s (fixed splits) or
// (P_b + s) * kt + hgv (balanced; P_b = splits of the sequences before b).
// A tile covers the output columns of its column block.
__global__ void __launch_bounds__(kAttnCombineThreads)
    gqa_attn_combine_kernel(const __grid_constant__ AttnCombineParams p) {
  constexpr int kBatch = 8;
  __shared__ float2 mz;                                      // (M, 1 / Z) of the head
  __shared__ float4 red[kAttnCombineThreads];                // per-part sums
  const int tile = blockIdx.x / p.heads;
  const int h = blockIdx.x - tile * p.heads;
  const int hgv = tile / p.B;
  const int b = tile - hgv * p.B;
  const int hg = hgv / p.ncol;
  const int DV = p.D / p.ncol;
  const int dv0 = (hgv - hg * p.ncol) * DV;
  int nsplit_b;
  size_t first, step;  // slot of split s: first + s * step
  if (!p.balanced) {
    const int L = clamped_len(p.seq_lens, b, p.Cmax);
    nsplit_b = L > 0 ? (L + p.rows_per_split - 1) / p.rows_per_split : 1;
    first = (size_t)tile * p.nsplit;
    step = 1;
  } else {
    const int sps = balanced_sps(p.seq_lens, p.B, p.Cmax, kAttnRows, p.kt, p.units);
    const int2 pn = balanced_prefix(p.seq_lens, p.Cmax, kAttnRows, sps, b);
    nsplit_b = pn.y;
    first = (size_t)pn.x * p.kt + hgv;
    step = p.kt;
  }
  grid_dependency_wait();
  grid_launch_dependents();
  if (nsplit_b <= 1) return;
  const int cols = DV / 4;
  const int parts = kAttnCombineThreads / cols;
  const int col = threadIdx.x % cols, part = threadIdx.x / cols;
  const int d = 4 * col;
  auto slot_of = [&](int s) { return (first + (size_t)s * step) * p.heads + h; };

  float4 x[kBatch];
  float em[kBatch];
  auto load = [&](int s0) {
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int s = s0 + u * parts;
      if (s < nsplit_b) {
        const size_t slot = slot_of(s);
        x[u] = __ldcg(reinterpret_cast<const float4*>(p.ws_o + slot * DV + d));
        em[u] = __ldcg(p.ws_ml + slot).x;
      }
    }
  };
  load(part);
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    float M = -INFINITY;
    for (int s = lane; s < nsplit_b; s += 32) M = fmaxf(M, __ldcg(p.ws_ml + slot_of(s)).x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float z = 0.0f;
    for (int s = lane; s < nsplit_b; s += 32) {
      const float2 v = __ldcg(p.ws_ml + slot_of(s));
      z = fmaf(v.y, exp2_fast(v.x - M), z);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    if (lane == 0) mz = make_float2(M, z > 0.0f ? 1.0f / z : 0.0f);
  }
  __syncthreads();
  const float2 hz = mz;
  float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  for (int s0 = part; s0 < nsplit_b; s0 += kBatch * parts) {
    if (s0 != part) load(s0);
#pragma unroll
    for (int u = 0; u < kBatch; ++u)
      if (s0 + u * parts < nsplit_b) {
        const float wgt = exp2_fast(em[u] - hz.x) * hz.y;
        acc.x = fmaf(x[u].x, wgt, acc.x);
        acc.y = fmaf(x[u].y, wgt, acc.y);
        acc.z = fmaf(x[u].z, wgt, acc.z);
        acc.w = fmaf(x[u].w, wgt, acc.w);
      }
  }
  red[threadIdx.x] = acc;
  __syncthreads();
  if (part == 0) {
    for (int q = 1; q < parts; ++q) add4(acc, red[q * cols + col]);
    *reinterpret_cast<float4*>(p.out + ((size_t)b * p.Hq + hg * p.heads + h) * p.D + dv0 + d) =
        acc;
  }
}

}  // namespace gqa_av
