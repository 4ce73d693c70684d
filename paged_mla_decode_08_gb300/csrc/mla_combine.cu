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
// One CTA of 128 threads per (job, query row): each thread owns 4 of the 512
// output columns, reads them from every split with 16-byte loads and writes
// 8 bytes of bf16.  Memory bound: traffic = nsplit * 2 KB + 1 KB per row.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "mla_internal.h"

namespace mla {

template <int CAP>
__global__ void __launch_bounds__(128) combine_kernel(const __grid_constant__ CombineList<CAP> jobs,
                                                      const __grid_constant__ DecodeArgs a) {
  const CombineJob job = jobs.job[blockIdx.x];
  const int m = blockIdx.y;
  const int M = a.rows;
  const float* plse = a.part_lse + (size_t)job.slot_begin * M + m;
  float mx = -CUDART_INF_F;
  for (int s = 0; s < job.nsplit; ++s) mx = fmaxf(mx, plse[(size_t)s * M]);
  const size_t row = (size_t)job.req * M + m;  // == (b*q_len + i)*H + h
  const int col = threadIdx.x * 4;
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out) + row * kLatent + col;
  if (mx == -CUDART_INF_F) {
    *reinterpret_cast<uint2*>(out) = make_uint2(0u, 0u);
    if (threadIdx.x == 0) a.lse[row] = -CUDART_INF_F;
    return;
  }
  float tot = 0.f;
  for (int s = 0; s < job.nsplit; ++s) tot += __expf(plse[(size_t)s * M] - mx);
  const float inv = 1.f / tot;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const float* po = a.part_o + ((size_t)job.slot_begin * M + m) * kLatent + col;
  for (int s = 0; s < job.nsplit; ++s) {
    const float l = plse[(size_t)s * M];
    if (l == -CUDART_INF_F) continue;
    const float wgt = __expf(l - mx) * inv;
    const float4 v = __ldg(reinterpret_cast<const float4*>(po + (size_t)s * M * kLatent));
    acc.x = fmaf(wgt, v.x, acc.x);
    acc.y = fmaf(wgt, v.y, acc.y);
    acc.z = fmaf(wgt, v.z, acc.z);
    acc.w = fmaf(wgt, v.w, acc.w);
  }
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
  uint2 pk;
  pk.x = *reinterpret_cast<uint32_t*>(&lo);
  pk.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(out) = pk;
  if (threadIdx.x == 0) a.lse[row] = mx + __logf(tot);
}

template <int CAP>
static cudaError_t launch_combine_cap(const std::vector<CombineJob>& jobs, const DecodeArgs& a,
                                      cudaStream_t stream) {
  CombineList<CAP> list;
  list.num_jobs = (int32_t)jobs.size();
  for (size_t i = 0; i < jobs.size(); ++i) list.job[i] = jobs[i];
  combine_kernel<CAP><<<dim3((unsigned)jobs.size(), (unsigned)a.rows), 128, 0, stream>>>(list, a);
  return cudaGetLastError();
}

cudaError_t launch_combine(const std::vector<CombineJob>& jobs, const DecodeArgs& a,
                           cudaStream_t stream) {
  if (jobs.empty()) return cudaSuccess;
  if (jobs.size() <= (size_t)kJobCapSmall) return launch_combine_cap<kJobCapSmall>(jobs, a, stream);
  return launch_combine_cap<kJobCapLarge>(jobs, a, stream);
}

}  // namespace mla
