// GQA AV decode reduction on the 5th-generation tensor cores (tcgen05) for
// sm_103a (GB300).
//
// Operation (page "pytorch/executorch pull 21063", summary paragraph):
//   out[b, q_h, d] = sum_{c < L_b} attn[b, c, q_h] * V[b, c, q_h / G, d].
//
// One CTA owns the same tile as the FMA kernel (head group, b, d-tile of up to
// 128 columns) and one context split of it, and reads each V row of its KV
// head from HBM once for all heads of the group. The splits are balanced over
// the batch: after the dependency wait every CTA reads all sequence lengths
// and cuts the batch's context rows into equal splits of whole stages (the
// length-balanced split helpers in gqa_av_kernel.cuh), so short sequences
// leave no CTA idle and every SM gets a like share of rows. Per pipeline stage of R
// context rows it computes the stage's contribution
//   D[m][n] = sum_k V[c0 + k][d0 + m] * attn[c0 + k][h0 + n]
// as one tcgen05 matrix product with M = 128 (output columns), N = the group's
// heads padded to a multiple of 16, K = R, accumulated in fp32 in tensor
// memory:
//   * A = V^T, read in place from the TMA-written stage: two 64-column halves
//     of R rows x 128 B in the 128-byte-swizzled MN-major layout.
//   * B = the weights, written by the converter warps as bf16 (fp16 for an
//     fp16 cache) in the K-major core-matrix layout. The fp32 weight w is
//     split as w = hi + lo with hi = round(w), lo = round(w - hi), and the
//     hi and lo rows of all heads form one B of 2N rows, so one MMA pass over
//     the stage's V gives both products: the weights keep about 16
//     significant bits (V is exact in its own type, and bf16 x bf16 /
//     fp16 x fp16 products are exact in fp32). fp16 weights are scaled by
//     2^12 first (exact, undone in the epilogue) so small weights do not fall
//     into fp16 subnormals.
//   * The stage's D (double-buffered in tensor memory, 2N columns: hi then
//     lo) is read back by the accumulator warps with tcgen05.ld and added
//     into fp32 registers, so the tensor core accumulates at most R/16
//     products into one value.
// Rows of a stage past the context are zeroed in shared memory (V) and given
// zero weight, so what lies there cannot reach the sum.
//
// Warp roles, each waiting only on its own inputs so the stages overlap:
// warps 0-3 accumulate (warp w reads tensor-memory lanes 32w..32w+31 = output
// columns), the next 2 or 4 warps write the weights of each stage as the B
// operand, then come the TMA producer warp and a warp that allocates tensor
// memory and one of whose threads issues the MMAs. With 2 converter warps the
// CTA's 8 warps spread evenly over the SM's four sub-partitions, so with at
// most 64 registers a thread (one 16-head block) four CTAs fit on an SM by
// registers; with 4 (10 warps) two do. The split combine is the FMA kernel's,
// reading one partial slot per CTA of this kernel. Every
// mbarrier wait is bounded; on expiry the CTA sets the device status word,
// lets its copies and MMAs in flight finish, frees its tensor memory and
// returns.
#pragma once

#include <type_traits>

#include "gqa_av_kernel.cuh"

namespace gqa_av {

constexpr int kMmaM = 128;         // output columns per MMA (D rows)
constexpr int kMmaAccWarps = 4;    // warps 0-3: one per tensor-memory lane quarter
constexpr int kMmaMaxCvtWarps = 4;  // weight-conversion warps: 2 or 4 (a plan choice)
constexpr int kMmaMaxThreads = 32 * (kMmaAccWarps + kMmaMaxCvtWarps + 2);
// Threads of a CTA with `cvt` converter warps (+ producer and MMA warps).
__host__ __device__ constexpr int mma_threads(int cvt) { return 32 * (kMmaAccWarps + cvt + 2); }
constexpr unsigned kErrMmaWait = 8u;

// tcgen05 shared-memory matrix descriptor: start address, leading- and
// stride-dimension byte offsets (all >> 4), the sm_100 descriptor version
// (bit 46) and the swizzle mode (bits 61-63: 0 none, 2 128-byte).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo,
                                              uint32_t swizzle) {
  return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) |
         (static_cast<uint64_t>(swizzle & 7u) << 61);
}

// Instruction descriptor of kind::f16: fp32 D, A and B of one 16-bit type
// (bf16 or fp16, never mixed), A MN-major, B K-major, N x M = n x 128.
template <typename Tag>
__host__ __device__ constexpr uint32_t mma_idesc(int n) {
  return (1u << 4) | (std::is_same<Tag, Bf16Tag>::value ? ((1u << 7) | (1u << 10)) : 0u) |
         (1u << 15) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(kMmaM >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05 operation this thread issued has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 16 consecutive fp32 columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Weights (a, b) split into 16-bit hi and lo pairs, each packed in a word
// (a in the low half) for the B operand.
__device__ __forceinline__ void split_weights(Bf16Tag, float a, float b, uint32_t& hi,
                                              uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(a - hf.x, b - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}
__device__ __forceinline__ void split_weights(Fp16Tag, float a, float b, uint32_t& hi,
                                              uint32_t& lo) {
  const float x = a * 4096.0f, y = b * 4096.0f;
  const __half2 h = __floats2half2_rn(x, y);
  const float2 hf = __half22float2(h);
  const __half2 l = __floats2half2_rn(x - hf.x, y - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}
__host__ __device__ constexpr float weight_unscale(Bf16Tag) { return 1.0f; }
__host__ __device__ constexpr float weight_unscale(Fp16Tag) { return 1.0f / 4096.0f; }

// Named barrier of the accumulator warps and the MMA warp: the warps that
// touch tensor memory.
__device__ __forceinline__ void mma_team_sync() {
  named_sync(2, 32 * (kMmaAccWarps + 1));
}

// Shared memory (offsets from a 1024-byte-aligned base):
//   [V ring: stages x R x 256 B, two 64-column halves of R x 128 B per stage]
//   [attn ring: stages x R x ap floats]
//   [B ring: stages x 2N (hi rows, then lo rows) x R x 2 B]
//   [mbarriers: full, empty, bready (kMaxStages each), dfull[2], dfree[2], drain]
//   [tensor-memory address] [the CTA's balanced split: 5 ints]
// The split of CTA blockIdx.x (length-balanced, see gqa_av_kernel.cuh).
struct MmaSplit {
  int b, c_begin, c_end, n_iters, alone;
  __device__ bool operator==(const MmaSplit& o) const {
    return b == o.b && c_begin == o.c_begin && c_end == o.c_end && n_iters == o.n_iters &&
           alone == o.alone;
  }
};

// Warp-collective. seq_lens null: every length is Cmax.
__device__ __forceinline__ MmaSplit mma_split(const int32_t* seq_lens, const Params& p, int K) {
  const int sps = balanced_sps(seq_lens, p.B, p.Cmax, p.R, K, p.split_units);
  const BalancedSplit bs =
      balanced_find(seq_lens, p.B, p.Cmax, p.R, sps, static_cast<int>(blockIdx.x) / K);
  MmaSplit r;
  r.b = bs.b;
  r.c_begin = bs.split * sps * p.R;
  r.c_end = min(r.c_begin + sps * p.R, bs.L);
  r.n_iters = bs.found ? max((r.c_end - r.c_begin + p.R - 1) / p.R, 1) : 0;
  r.alone = bs.n == 1;
  return r;
}

// Lengths a lane keeps in registers: batches of up to 256 sequences find
// their split from one round of loads.
constexpr int kLenRegs = 8;

__device__ __forceinline__ void load_lens(const int32_t* seq_lens, int B, int Cmax,
                                          int (&L)[kLenRegs]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 0; j < kLenRegs; ++j) {
    const int b = 32 * j + lane;
    L[j] = b < B ? clamped_len(seq_lens, b, Cmax) : 0;
  }
}

// mma_split from lengths in registers (B <= 32 * kLenRegs). Warp-collective.
__device__ __forceinline__ MmaSplit split_from_lens(const int (&L)[kLenRegs], const Params& p,
                                                    int K) {
  const int lane = threadIdx.x & 31;
  long long s = 0;
#pragma unroll
  for (int j = 0; j < kLenRegs; ++j) s += (L[j] + p.R - 1) / p.R;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  const long long sps_l = (s * K + p.split_units - 1) / p.split_units;
  const int sps = sps_l > 1 ? static_cast<int>(sps_l) : 1;
  const int q = static_cast<int>(blockIdx.x) / K;
  int base = 0, hb = -1, hL = 0, hn = 0, hsplit = 0;
#pragma unroll
  for (int j = 0; j < kLenRegs; ++j) {
    if (32 * j < p.B && hb < 0) {  // warp-uniform
      const int n = 32 * j + lane < p.B ? balanced_splits_of(L[j], p.R, sps) : 0;
      int incl = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      const unsigned hit =
          __ballot_sync(0xffffffffu, n > 0 && q >= base + incl - n && q < base + incl);
      if (hit) {
        const int src = __ffs(hit) - 1;
        hb = 32 * j + src;
        hL = __shfl_sync(0xffffffffu, L[j], src);
        hn = __shfl_sync(0xffffffffu, n, src);
        hsplit = q - base - __shfl_sync(0xffffffffu, incl - n, src);
      }
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  MmaSplit r{0, 0, 0, 0, 0};
  if (hb >= 0) {
    r.b = hb;
    r.c_begin = hsplit * sps * p.R;
    r.c_end = min(r.c_begin + sps * p.R, hL);
    r.n_iters = max((r.c_end - r.c_begin + p.R - 1) / p.R, 1);
    r.alone = hn == 1;
  }
  return r;
}

template <typename Tag, int NB>
__global__ void __launch_bounds__(kMmaMaxThreads, NB == 1 ? 3 : (NB == 2 ? 2 : 1))
    gqa_av_mma_kernel(const __grid_constant__ Params p) {
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
      mbar_init(empty0 + 8 * s, 1);                     // one tcgen05.commit per stage
      mbar_init(bready0 + 8 * s, cvt_warps);            // one arrival per converter warp
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

  // The CTA's tile and context split. Fixed splits (p.balanced == 0): CTA
  // (tile, split) = (blockIdx / nsplit, blockIdx % nsplit), split s covering
  // rows [s * rows_per_split, (s + 1) * rows_per_split) of its sequence, so
  // the first stages can be issued before the length is read, and every warp
  // reads the one length it needs itself. Balanced splits: tile k = blockIdx
  // % K of a sequence the batch's lengths decide (length-balanced split
  // helpers in gqa_av_kernel.cuh); the producer warp works the split out and
  // hands it to the other warps through shared memory at named barrier 3.
  // A CTA with no context rows has n_iters 0.
  const int K = p.hgroups * p.ndt;
  int hg, dti, tile = 0, split = 0;
  if (p.balanced) {
    const int k = blockIdx.x % K;
    hg = k / p.ndt;
    dti = k - hg * p.ndt;
  } else {
    tile = blockIdx.x / p.nsplit;
    split = blockIdx.x - tile * p.nsplit;
    hg = tile / (p.B * p.ndt);
    dti = tile - hg * (p.B * p.ndt);
    dti -= (dti / p.ndt) * p.ndt;
  }
  const int h0 = hg * p.heads;
  const int kv_h = h0 / p.G;
  const int d0 = dti * p.dt;
  const int a_shift = p.attn_tma ? (h0 & 3) : 0;
  const int b_fixed = p.balanced ? 0 : (tile - hg * (p.B * p.ndt)) / p.ndt;
  int* split_info = reinterpret_cast<int*>(bars + 3 * kMaxStages + 6);
  // The fixed split of this CTA once the sequence length is known.
  auto fixed_split = [&](MmaSplit& f) {
    const int L = clamped_len(p.seq_lens, b_fixed, p.Cmax);
    const int nsplit_b = L > 0 ? (L + p.rows_per_split - 1) / p.rows_per_split : 1;
    f.b = b_fixed;
    f.c_begin = split * p.rows_per_split;
    f.c_end = min(f.c_begin + p.rows_per_split, L);
    f.n_iters = split < nsplit_b ? max((f.c_end - f.c_begin + p.R - 1) / p.R, 1) : 0;
    f.alone = nsplit_b == 1;
    return tile * p.nsplit + split;
  };

  grid_dependency_wait();
  grid_launch_dependents();

  if (warp == producer_warp) {
    // ----------------------------------------------------------------- producer
    const int per_row = p.heads / p.avec;
    auto issue = [&](int stage, int b, int c0, int rows) {
      const uint32_t full = full0 + 8 * stage;
      const uint32_t vdst = vring_s + (uint32_t)stage * p.v_stage_bytes;
      if (p.block_table) {
        // Paged: the stage's block indices loaded by the lanes together (lane
        // j for box j), then lane 0 issues one box a block and V half.
        const int nbox = p.R / p.chunk_rows;  // <= 32
        const int2 mine = lane < nbox ? v_row_coord(p, b, c0 + lane * p.chunk_rows) : make_int2(0, 0);
        if (lane == 0)
          mbar_arrive_expect_tx(full, (uint32_t)p.v_halves * (p.v_stage_bytes / 2) +
                                          (p.attn_tma ? p.a_stage_bytes : 0u));
        for (int j = 0; j < nbox; ++j) {
          const int rx = __shfl_sync(0xffffffffu, mine.x, j);
          const int ry = __shfl_sync(0xffffffffu, mine.y, j);
          if (lane == 0)
            for (int h = 0; h < p.v_halves; ++h)
              tma_load_4d(vdst + (uint32_t)h * p.v_stage_bytes / 2 + (uint32_t)(j * p.chunk_rows) * 128,
                          &p.v_map, d0 + 64 * h, kv_h, rx, ry, full, policy);
        }
      }
      if (lane == 0) {
        if (!p.block_table) {
          mbar_arrive_expect_tx(full, (uint32_t)p.v_halves * (p.v_stage_bytes / 2) +
                                          (p.attn_tma ? p.a_stage_bytes : 0u));
          for (int h = 0; h < p.v_halves; ++h)
            tma_load_4d(vdst + (uint32_t)h * p.v_stage_bytes / 2, &p.v_map, d0 + 64 * h, kv_h, c0,
                        b, full, policy);
        }
        if (p.attn_tma)
          tma_load_3d(aring_s + (uint32_t)stage * p.a_stage_bytes, &p.a_map, h0 - a_shift, c0, b,
                      full, policy);
      }
      if (p.attn_tma) return;
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
    };

    MmaSplit f;
    int pre = 0;
    if (!p.balanced) {
      // The first stage(s) go out before the length is read.
      const int c_begin = split * p.rows_per_split;
      pre = min(min(min(p.early_stages, p.stages), p.rows_per_split / p.R),
                (p.Cmax - c_begin + p.R - 1) / p.R);
      for (int it = 0; it < pre; ++it) {
        const int c0 = c_begin + it * p.R;
        issue(it, b_fixed, c0, min(p.R, p.Cmax - c0));
      }
      fixed_split(f);
    } else {
      if (p.B <= 32 * kLenRegs) {
        int lens[kLenRegs];
        load_lens(p.seq_lens, p.B, p.Cmax, lens);
        f = split_from_lens(lens, p, K);
      } else {
        f = mma_split(p.seq_lens, p, K);
      }
      if (lane == 0) {
        split_info[0] = f.b;
        split_info[1] = f.c_begin;
        split_info[2] = f.c_end;
        split_info[3] = f.n_iters;
        split_info[4] = f.alone;
      }
      named_arrive(3, blockDim.x);
    }

    int issued = pre;
    bool ok = true;
    for (int it = pre; it < f.n_iters; ++it) {
      const int stage = it % p.stages;
      const uint32_t parity = ((it / p.stages) & 1) ^ 1;  // a fresh slot passes at once
      if (!mbar_wait(empty0 + 8 * stage, parity, p.timeout_ns)) {
        atomicOr(p.status, kErrEmptyWait);
        ok = false;
        break;
      }
      const int c0 = f.c_begin + it * p.R;
      issue(stage, f.b, c0, min(p.R, f.c_end - c0));
      issued = it + 1;
    }
    cp_async_wait_all();
    if (!ok) {
      for (int it = max(0, issued - p.stages); it < issued; ++it)
        if (!mbar_wait(full0 + 8 * (it % p.stages), (it / p.stages) & 1, p.timeout_ns))
          atomicOr(p.status, kErrDrain);
    }
    // Early stages past the split's context (a split past its length): let
    // them land before the CTA exits.
    for (int it = f.n_iters; it < pre; ++it)
      if (!mbar_wait(full0 + 8 * it, 0, p.timeout_ns) && lane == 0) atomicOr(p.status, kErrDrain);
    return;
  }

  MmaSplit f;
  int slot;
  if (!p.balanced) {
    slot = fixed_split(f);
  } else {
    named_sync(3, blockDim.x);
    f.b = split_info[0];
    f.c_begin = split_info[1];
    f.c_end = split_info[2];
    f.n_iters = split_info[3];
    f.alone = split_info[4];
    slot = blockIdx.x;
  }
  const int b = f.b, c_begin = f.c_begin, c_end = f.c_end, n_iters = f.n_iters, alone = f.alone;

  const uint32_t b_half = (uint32_t)N * p.R * 2;   // bytes of one of hi / lo

  if (warp == issuer_warp) {
    // -------------------------------------------------------------- MMA issuer
    const uint32_t idesc = mma_idesc<Tag>(2 * N);
    const uint32_t a_lbo = (uint32_t)p.R * 128;      // second 64-column half
    const uint32_t b_sbo = (uint32_t)(p.R / 8) * 128;  // next 8 rows of B
    bool ok = true;
    if (lane == 0) {
      int issued = 0;
      for (int it = 0; it < n_iters; ++it) {
        const int stage = it % p.stages, j = it & 1;
        if (!mbar_poll(bready0 + 8 * stage, (it / p.stages) & 1, p.timeout_ns) ||
            (it >= 2 && !mbar_poll(dfree0 + 8 * j, ((it - 2) >> 1) & 1, p.timeout_ns))) {
          atomicOr(p.status, kErrMmaWait);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(j * 2 * N);
        const uint32_t a0 = vring_s + (uint32_t)stage * p.v_stage_bytes;
        const uint32_t bb = bring_s + (uint32_t)stage * 2 * b_half;
        // K step kk starts 16 rows on: 2048 B into each V half, two core
        // matrices (256 B) into B. The start-address field holds address / 16
        // in its low 14 bits, so the step is added to the descriptor itself.
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
      }
      if (issued > 0) {
        mma_commit(drain);
        if (!mbar_wait(drain, 0, p.timeout_ns)) atomicOr(p.status, kErrMmaWait);
      }
    }
    (void)ok;
    __syncwarp();
    mma_team_sync();  // consumers are done with tensor memory
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
    for (int it = 0; it < n_iters; ++it) {
      const int stage = it % p.stages;
      if (!mbar_poll(full0 + 8 * stage, (it / p.stages) & 1, p.timeout_ns)) {
        atomicOr(p.status, kErrFullWait);
        break;
      }
      const int c0 = c_begin + it * p.R;
      const int valid = min(p.R, c_end - c0);
      const float* ast = aring + (size_t)stage * p.R * p.ap + a_shift;
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
    }
    return;
  }

  // -------------------------------------------------------------- accumulators
  // Thread t owns output column m = t (tensor-memory lane t) of every head.
  const int m = tid;
  float acc[N];
#pragma unroll
  for (int n = 0; n < N; ++n) acc[n] = 0.0f;
  bool ok = true;
  for (int it = 0; it < n_iters; ++it) {   // add stage it's D into acc, free its buffer
    const int j = it & 1;
    if (!mbar_wait(dfull0 + 8 * j, (it >> 1) & 1, p.timeout_ns)) {
      atomicOr(p.status, kErrMmaWait);
      ok = false;
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
  }

  if (ok && n_iters > 0) {
    const float unscale = weight_unscale(Tag{});
    const int tile_elems = p.heads * p.dt;
    float* part = p.ws + (size_t)slot * tile_elems;
    if (m < p.dt && d0 + m < p.D) {
#pragma unroll
      for (int n = 0; n < N; ++n) {
        if (n < p.heads) {
          const float v = acc[n] * unscale;
          if (alone) p.out[((size_t)b * p.Hq + h0 + n) * p.D + d0 + m] = v;
          else __stcg(part + (size_t)n * p.dt + m, v);
        }
      }
    }
  }
  tc_fence_before();
  mma_team_sync();
}

// Launch and occupancy of one instantiation (defined with the instantiations).
template <typename Tag, int NB>
cudaError_t launch_mma(const Params& p, int grid, int smem_bytes, cudaStream_t stream);
template <typename Tag, int NB>
cudaError_t occupancy_mma(int smem_limit, int smem_bytes, int* ctas_per_sm);

}  // namespace gqa_av
