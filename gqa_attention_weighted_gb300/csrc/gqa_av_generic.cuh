// The AV reduction for any head dimension and element-aligned pointers.
//
//   out[b, q_h, d] = sum_{c < L_b} attn[b, c, q_h] * V[b, c, q_h / G, d]
//
// (page "pytorch/executorch pull 21063", summary paragraph), with the same
// GQA-reuse grouping as the main kernels: a CTA owns the query heads of one KV
// head, so each V element is loaded once for all of them. The main kernels
// move V by TMA boxes and 16-byte vectors, which needs D % 8 == 0 and 16-byte
// aligned attn, V and out. The page's own granularity is a 4-wide texel, and
// callers may hand over sub-views of larger buffers; this kernel takes every
// D >= 1 and pointers aligned only to their element type, with plain loads:
//
// gqa_av_generic_kernel: CTA (tile = (head group, b), context split) of 256
// threads (about eight CTAs per SM), a thread per (row slot, column) over
// column blocks of up to 256.
// Consecutive threads read consecutive V elements of one row (2-byte loads,
// coalesced); the weights of a row are the same for every thread (broadcast
// loads). Heads go in passes of 8 fp32 accumulators. The row slots are summed
// in slot order through shared memory; a sequence that fits one split writes
// out, otherwise each split writes its partial and gqa_av_generic_combine
// sums the splits in a fixed order. Results are bitwise reproducible.
#pragma once

#include "gqa_av_kernel.cuh"

namespace gqa_av {

constexpr int kGenThreads = 256;
constexpr int kGenHeads = 8;  // fp32 accumulators a thread keeps per pass

struct GenericParams {
  const float* attn;        // [B, Cmax, Hq], 4-byte aligned
  const uint16_t* v;        // [B, Cmax, Hkv, D] bf16 / fp16 bits, 2-byte aligned
  const int32_t* seq_lens;  // [B] or null
  float* out;               // [B, Hq, D], 4-byte aligned
  float* ws;                // [tiles][nsplit][heads][D] split partials
  int B, Cmax, Hq, Hkv, D, G;
  int heads, hgroups;       // query heads per CTA, Hq / heads
  int cw, row_par;          // columns per block (<= 256), row slots (256 / cw)
  int rows_per_split, nsplit;
};

__device__ __forceinline__ float widen1(Bf16Tag, uint16_t x) {
  return __uint_as_float(static_cast<uint32_t>(x) << 16);
}
__device__ __forceinline__ float widen1(Fp16Tag, uint16_t x) {
  return __half2float(__ushort_as_half(x));
}

template <typename Tag>
__global__ void __launch_bounds__(kGenThreads) gqa_av_generic_kernel(const GenericParams p) {
  __shared__ float red[kGenHeads * kGenThreads];
  const int tile = blockIdx.x / p.nsplit;
  const int split = blockIdx.x - tile * p.nsplit;
  const int hg = tile / p.B;
  const int b = tile - hg * p.B;
  const int h0 = hg * p.heads;
  const int kv_h = h0 / p.G;
  const int L = clamped_len(p.seq_lens, b, p.Cmax);
  const int nsplit_b = L > 0 ? (L + p.rows_per_split - 1) / p.rows_per_split : 1;
  if (split >= nsplit_b) return;  // uniform over the CTA
  const int c_begin = split * p.rows_per_split;
  const int c_end = min(c_begin + p.rows_per_split, L);
  const int col = threadIdx.x % p.cw;
  const int rs = threadIdx.x / p.cw;
  const size_t v_row = (size_t)p.Hkv * p.D;  // elements between consecutive positions
  const uint16_t* vb = p.v + ((size_t)b * p.Cmax * p.Hkv + kv_h) * p.D;
  const float* ab = p.attn + (size_t)b * p.Cmax * p.Hq + h0;

  for (int d0 = 0; d0 < p.D; d0 += p.cw) {
    const int d = d0 + col;
    const bool active = rs < p.row_par && d < p.D;
    for (int g0 = 0; g0 < p.heads; g0 += kGenHeads) {
      const int ng = min(kGenHeads, p.heads - g0);
      float acc[kGenHeads];
#pragma unroll
      for (int g = 0; g < kGenHeads; ++g) acc[g] = 0.0f;
      if (active) {
        const uint16_t* vp = vb + d;
        const float* ap = ab + g0;
#pragma unroll 8
        for (int c = c_begin + rs; c < c_end; c += p.row_par) {
          const float x = widen1(Tag{}, vp[(size_t)c * v_row]);
          const float* a = ap + (size_t)c * p.Hq;
#pragma unroll
          for (int g = 0; g < kGenHeads; ++g)
            if (g < ng) acc[g] = fmaf(a[g], x, acc[g]);
        }
      }
      __syncthreads();  // the previous pass has read `red`
      if (rs < p.row_par) {
#pragma unroll
        for (int g = 0; g < kGenHeads; ++g) red[(g * p.row_par + rs) * p.cw + col] = acc[g];
      }
      __syncthreads();
      if (rs == 0 && d < p.D) {
        for (int g = 0; g < ng; ++g) {
          float s = 0.0f;
          for (int r = 0; r < p.row_par; ++r) s += red[(g * p.row_par + r) * p.cw + col];
          if (nsplit_b == 1)
            p.out[((size_t)b * p.Hq + h0 + g0 + g) * p.D + d] = s;
          else
            __stcg(p.ws + (((size_t)tile * p.nsplit + split) * p.heads + g0 + g) * p.D + d, s);
        }
      }
    }
  }
}

// CTA per (tile, 32 consecutive outputs): 8 parts of 32 threads, part r
// summing splits r, r + 8, ... in order; the parts are then added in part
// order, so the result is deterministic. Launched after the main kernel on
// the same stream.
constexpr int kGenCombineOut = 32;
__global__ void __launch_bounds__(kGenThreads) gqa_av_generic_combine(const GenericParams p) {
  __shared__ float red[kGenThreads];
  constexpr int kParts = kGenThreads / kGenCombineOut;
  const int n = p.heads * p.D;
  const int chunks = (n + kGenCombineOut - 1) / kGenCombineOut;
  const int tile = blockIdx.x / chunks;
  const int chunk = blockIdx.x - tile * chunks;
  const int hg = tile / p.B;
  const int b = tile - hg * p.B;
  const int L = clamped_len(p.seq_lens, b, p.Cmax);
  const int nsplit_b = L > 0 ? (L + p.rows_per_split - 1) / p.rows_per_split : 1;
  if (nsplit_b <= 1) return;  // written by the main kernel
  const int e = chunk * kGenCombineOut + (threadIdx.x % kGenCombineOut);
  const int part = threadIdx.x / kGenCombineOut;
  const float* src = p.ws + (size_t)tile * p.nsplit * n;
  float s = 0.0f;
  if (e < n) {
#pragma unroll 4
    for (int sp = part; sp < nsplit_b; sp += kParts) s += __ldcg(src + (size_t)sp * n + e);
  }
  red[threadIdx.x] = s;
  __syncthreads();
  if (part == 0 && e < n) {
    for (int r = 1; r < kParts; ++r) s += red[r * kGenCombineOut + threadIdx.x];
    const int h = e / p.D, d = e - h * p.D;
    p.out[((size_t)b * p.Hq + hg * p.heads + h) * p.D + d] = s;
  }
}

}  // namespace gqa_av
