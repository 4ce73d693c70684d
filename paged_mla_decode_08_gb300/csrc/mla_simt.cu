// Plain SIMT split-KV decode kernel: one CTA per (segment, query row).
//
// This is the simple, obviously-correct CUDA path: each warp walks every 4th
// visible key of the segment, reads the 576-wide cache row through the block
// table (one page lookup per key), forms the score with a warp reduction and
// keeps an online softmax (running max, running sum, 512-wide accumulator
// spread over the lanes); the four warps are merged through shared memory at
// the end.  It re-reads the segment's keys once per query row (through L2)
// and uses CUDA cores only, so it is far from the roofline; the tensor-core
// kernel in mla_sm103.cu is the fast path.  Both consume the same schedule
// and write the same outputs / partials.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "mla_internal.h"

namespace mla {

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
  return __uint_as_float((uint32_t)b << 16);
}

// Exact e4m3fn -> fp32: place the 7 magnitude bits where an fp32 exponent /
// mantissa pair starts (exponent bias 127 instead of 7), then rescale by
// 2^(127-7) = 2^120.  Exponent-field-0 codes land on fp32 subnormals and are
// rescaled exactly as well (this file is built without flush-to-zero).  The
// NaN code is not special-cased: rows that may hold it are never read.
__device__ __forceinline__ float e4m3_bits_to_f32(uint32_t x) {
  const uint32_t bits = ((x & 0x7Fu) << 20) | ((x & 0x80u) << 24);
  return __uint_as_float(bits) * 0x1p120f;
}

template <int CAP>
__global__ void __launch_bounds__(128) simt_decode_kernel(const __grid_constant__ Schedule<CAP> sched,
                                                          const __grid_constant__ DecodeArgs a) {
  const Segment sg = sched.seg[blockIdx.x];
  const int m = blockIdx.y;
  const int H = a.num_heads;
  const int b = sg.req;
  const int i = m / H;
  const int h = m % H;
  const int tok = b * a.q_len + i;
  const int L = a.seq_lens[b];
  const int vis = L - a.q_len + 1 + i;
  const int j0 = sg.tile_begin * kTileTokens;
  // never past the block-table row, whatever the device lengths say
  const int j1 = min(min(sg.tile_end * kTileTokens, vis), a.bt_stride * a.page_size);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  __shared__ float q_s[kKvDim];
  __shared__ float o_s[4][kLatent];
  __shared__ float m_s[4], l_s[4];

  const uint16_t* qn = reinterpret_cast<const uint16_t*>(a.q_nope) + ((size_t)tok * H + h) * kLatent;
  const uint16_t* qp = reinterpret_cast<const uint16_t*>(a.q_pe) + ((size_t)tok * H + h) * kRope;
  for (int d = threadIdx.x; d < kKvDim; d += 128)
    q_s[d] = d < kLatent ? bf16_bits_to_f32(qn[d]) : bf16_bits_to_f32(qp[d - kLatent]);
  __syncthreads();

  float run_m = -CUDART_INF_F, run_l = 0.f;
  float o[16];
#pragma unroll
  for (int c = 0; c < 16; ++c) o[c] = 0.f;

  const int32_t* bt = a.block_table + (size_t)b * a.bt_stride;
  for (int j = j0 + warp; j < j1; j += 4) {
    const int page = bt[j / a.page_size];
    if (page < 0 || page >= a.num_pages) continue;  // invalid id: key skipped
    const size_t row = (size_t)page * a.page_size + (j % a.page_size);
    float v[18];
    if (a.kv_dtype == 0) {
      const uint16_t* r = reinterpret_cast<const uint16_t*>(a.kv) + row * kKvDim;
#pragma unroll
      for (int k = 0; k < 18; ++k) v[k] = bf16_bits_to_f32(r[lane + 32 * k]);
    } else {
      const uint8_t* r = reinterpret_cast<const uint8_t*>(a.kv) + row * kKvDim;
#pragma unroll
      for (int k = 0; k < 18; ++k) v[k] = e4m3_bits_to_f32(r[lane + 32 * k]);
    }
    float dot = 0.f;
#pragma unroll
    for (int k = 0; k < 18; ++k) dot = fmaf(v[k], q_s[lane + 32 * k], dot);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
    const float s = dot * a.score_scale_log2;
    const float mn = fmaxf(run_m, s);
    const float corr = exp2f(run_m - mn);
    const float p = exp2f(s - mn);
    run_l = run_l * corr + p;
#pragma unroll
    for (int c = 0; c < 16; ++c) o[c] = fmaf(o[c], corr, p * v[c]);
    run_m = mn;
  }
#pragma unroll
  for (int c = 0; c < 16; ++c) o_s[warp][lane + 32 * c] = o[c];
  if (lane == 0) { m_s[warp] = run_m; l_s[warp] = run_l; }
  __syncthreads();

  float M = fmaxf(fmaxf(m_s[0], m_s[1]), fmaxf(m_s[2], m_s[3]));
  float wgt[4], l = 0.f;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    wgt[w] = (M == -CUDART_INF_F) ? 0.f : exp2f(m_s[w] - M);
    l += wgt[w] * l_s[w];
  }
  const size_t orow = (size_t)b * a.rows + m;
  const bool empty = !(l > 0.f);
  const float inv = empty ? 0.f : a.out_scale / l;
  const float lse = empty ? -CUDART_INF_F : (M + log2f(l)) * 0.6931471805599453f;
  for (int c = threadIdx.x; c < kLatent; c += 128) {
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) acc = fmaf(wgt[w], o_s[w][c], acc);
    acc *= inv;
    if (sg.slot < 0)
      reinterpret_cast<__nv_bfloat16*>(a.out)[orow * kLatent + c] = __float2bfloat16_rn(acc);
    else
      a.part_o[(((size_t)sg.slot * (kLatent / 4) + c / 4) * a.rows + m) * 4 + (c & 3)] = acc;  // chunk-major
  }
  if (threadIdx.x == 0) {
    if (sg.slot < 0) a.lse[orow] = lse;
    else a.part_lse[(size_t)sg.slot * a.rows + m] = lse;
  }
}

template <int CAP>
static cudaError_t launch_simt_cap(const mla_plan& p, const DecodeArgs& a, cudaStream_t stream) {
  Schedule<CAP> s;
  s.num_workers = p.num_workers;
  s.num_segments = (int32_t)p.segs.size();
  for (int w = 0; w <= p.num_workers; ++w) s.worker_seg[w] = p.worker_seg[w];
  for (size_t i = 0; i < p.segs.size(); ++i) s.seg[i] = p.segs[i];
  simt_decode_kernel<CAP><<<dim3((unsigned)p.segs.size(), (unsigned)a.rows), 128, 0, stream>>>(s, a);
  return cudaGetLastError();
}

cudaError_t launch_simt(const mla_plan& p, const DecodeArgs& a, cudaStream_t stream) {
  if (p.segs.size() <= (size_t)kSegCapSmall) return launch_simt_cap<kSegCapSmall>(p, a, stream);
  return launch_simt_cap<kSegCapLarge>(p, a, stream);
}

}  // namespace mla
