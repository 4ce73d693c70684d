// LSE combine: merges the per-split partial results of split requests.
//
// A request cut into k segments has k partial rows per query row m:
// O_s = (sum_j p_j c_kv_j) / l_s (already scaled by the value
// dequantisation factor) and lse_s.  The merge is
//     lse = ln sum_s e^{lse_s},   out = sum_s e^{lse_s - lse} O_s,
// where a split that saw no visible key has lse_s = -inf and weighs nothing;
// if every split is empty the row is out = 0, lse = -inf, as the zero-KV rows
// of the pages (sglang trtllm_mla_backend.py, forward_extend: fixed-up rows
// with lse = -inf so the merge ignores them).
//
// Partials are chunk-major, part_o[slot][c][row] (c = 16-byte chunk of 4
// output columns), so that the producing kernels store coalesced.  One CTA of
// 256 threads per (job, block of 32 query rows, quarter of the 128 chunks):
// the split weights e^{lse_s - lse} of the 32 rows go to shared memory, then
// a warp owns 4 chunks and reads them for 32 consecutive rows (512
// contiguous bytes per chunk and split, four independent loads in flight),
// and the 32 x 128 bf16 result is transposed through shared memory so that
// each output row segment is written with contiguous 16-byte stores.
// Memory bound: nsplit * 2 KB read + 1 KB written per row.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "mla_internal.h"

namespace mla {

constexpr int kCombRows = 32;
constexpr int kCombChunks = 32;  // per CTA: a quarter of the 128 chunks

template <int CAP>
__global__ void __launch_bounds__(256) combine_kernel(const __grid_constant__ CombineList<CAP> jobs,
                                                      const __grid_constant__ DecodeArgs a) {
  extern __shared__ float s_w[];  // [nsplit][32] weights (0 for -inf splits)
  const CombineJob job = jobs.job[blockIdx.x];
  const int M = a.rows;
  const int r0 = blockIdx.y * kCombRows;
  const int c0 = blockIdx.z * kCombChunks;
  const int nrows = min(kCombRows, M - r0);
  __shared__ uint2 s_out[kCombRows][kCombChunks + 1];

  if (threadIdx.x < kCombRows) {
    const int r = threadIdx.x;
    float mx = -CUDART_INF_F, tot = 0.f;
    const float* pl = a.part_lse + (size_t)job.slot_begin * M + r0 + r;
    if (r < nrows) {
      for (int s = 0; s < job.nsplit; ++s) mx = fmaxf(mx, pl[(size_t)s * M]);
      if (mx != -CUDART_INF_F)
        for (int s = 0; s < job.nsplit; ++s) tot += __expf(pl[(size_t)s * M] - mx);
      if (blockIdx.z == 0) a.lse[(size_t)job.req * M + r0 + r] = tot > 0.f ? mx + __logf(tot) : -CUDART_INF_F;
    }
    const float inv = tot > 0.f ? 1.f / tot : 0.f;
    for (int s = 0; s < job.nsplit; ++s) {
      const float l = r < nrows ? pl[(size_t)s * M] : -CUDART_INF_F;
      s_w[s * kCombRows + r] = (inv > 0.f && l != -CUDART_INF_F) ? __expf(l - mx) * inv : 0.f;
    }
  }
  __syncthreads();

  const int r = threadIdx.x & 31;  // row within the block
  const int cw = threadIdx.x >> 5;  // warp: chunks c0 + cw + 8k, k < 4
  float4 acc[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (r < nrows) {
    const float4* po = reinterpret_cast<const float4*>(a.part_o) +
                       ((size_t)job.slot_begin * (kLatent / 4) + c0 + cw) * M + r0 + r;
    const size_t split_stride = (size_t)(kLatent / 4) * M;
    for (int s = 0; s < job.nsplit; ++s) {
      const float wgt = s_w[s * kCombRows + r];
      if (wgt == 0.f) continue;
      float4 v[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) v[k] = __ldg(po + s * split_stride + (size_t)(8 * k) * M);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        acc[k].x = fmaf(wgt, v[k].x, acc[k].x);
        acc[k].y = fmaf(wgt, v[k].y, acc[k].y);
        acc[k].z = fmaf(wgt, v[k].z, acc[k].z);
        acc[k].w = fmaf(wgt, v[k].w, acc[k].w);
      }
    }
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc[k].x, acc[k].y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc[k].z, acc[k].w);
    s_out[r][cw + 8 * k] = make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
  }
  __syncthreads();
  // 32 rows x 256 bytes: a half-warp writes one row segment (16 lanes x 16 B)
  const int hw = threadIdx.x >> 4, l16 = threadIdx.x & 15;
  for (int rr = hw; rr < nrows; rr += 16) {
    const size_t row = (size_t)job.req * M + r0 + rr;
    uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) + row * kLatent + 4 * c0) + l16;
    const uint2 x0 = s_out[rr][2 * l16], x1 = s_out[rr][2 * l16 + 1];
    *dst = make_uint4(x0.x, x0.y, x1.x, x1.y);
  }
}

template <int CAP>
static cudaError_t launch_combine_cap(const std::vector<CombineJob>& jobs, const DecodeArgs& a,
                                      cudaStream_t stream) {
  CombineList<CAP> list;
  list.num_jobs = (int32_t)jobs.size();
  for (size_t i = 0; i < jobs.size(); ++i) list.job[i] = jobs[i];
  int maxsplit = 1;
  for (const CombineJob& j : jobs) maxsplit = j.nsplit > maxsplit ? j.nsplit : maxsplit;
  const size_t smem = (size_t)maxsplit * kCombRows * sizeof(float);  // <= 128 splits: 16 KB
  combine_kernel<CAP><<<dim3((unsigned)jobs.size(), (unsigned)((a.rows + kCombRows - 1) / kCombRows),
                             (unsigned)(kLatent / 4 / kCombChunks)),
                        256, smem, stream>>>(list, a);
  return cudaGetLastError();
}

cudaError_t launch_combine(const std::vector<CombineJob>& jobs, const DecodeArgs& a,
                           cudaStream_t stream) {
  if (jobs.empty()) return cudaSuccess;
  if (jobs.size() <= (size_t)kJobCapSmall) return launch_combine_cap<kJobCapSmall>(jobs, a, stream);
  return launch_combine_cap<kJobCapLarge>(jobs, a, stream);
}

}  // namespace mla
