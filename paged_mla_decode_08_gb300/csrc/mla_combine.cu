// LSE combine: merges the per-split partial results of split requests.
//
// A request cut into k segments has k partial rows per query row m:
// O_s = (sum_j p_j c_kv_j) / l_s (already scaled by the value
// dequantisation factor) and lse_s.  The merge is
//     lse = ln sum_s e^{lse_s},   out = sum_s e^{lse_s - lse} O_s,
// where a split that saw no visible key has lse_s = -inf and weighs nothing
// (a split with lse_s = NaN makes the row NaN, as the definition does);
// if every split is empty the row is out = 0, lse = -inf, as the zero-KV rows
// of the pages (sglang trtllm_mla_backend.py, forward_extend: fixed-up rows
// with lse = -inf so the merge ignores them).
//
// Partials are bf16 and chunk-major, part_o[slot][c][row] (c = 16-byte chunk
// of 8 output columns), so that the producing kernel stores coalesced.  One
// CTA of 256 threads per (job, block of 32 query rows, quarter of the 64
// chunks): a warp owns 2 chunks and reads them for 32 consecutive rows (512
// contiguous bytes per chunk and split).  A launch whose widest job has more
// than 8 splits gives each CTA a sixteenth of the row instead (128 threads, a
// chunk per warp), so a request split 40 ways is merged by 64 CTAs per 128
// rows, not 16.  The partials of the first 4, 8 or 16
// splits (a group sized for the widest job of the launch) are requested
// before the split weights e^{lse_s - lse} are computed (one warp, into
// shared memory), so both memory latencies overlap, and later groups are
// loaded one round each; the
// 32-row result is transposed through shared memory so that each
// output row segment is written with contiguous 16-byte stores.  The bf16
// partials add one rounding of O_s (relative 2^-9) before the merge, well
// inside the output tolerance, and halve the bytes written and read.
// Memory bound: nsplit * 1 KB read + 1 KB written per row.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "mla_internal.h"

namespace mla {

constexpr int kCombRows = 32;
constexpr int kChunkCols = 8;                  // a 16-byte chunk of bf16 partial outputs
constexpr int kChunks = kLatent / kChunkCols;  // 64 per row
constexpr int kCombChunks = kChunks / 4;       // per CTA: a quarter of the row

__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
// max(a, b), NaN if either is NaN
__device__ __forceinline__ float max_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

// One (job, 32-row block, 1/kParts of the columns) of the merge; called after
// the grid dependency wait.  kGroup splits' partials are in flight at a time:
// the merge is a chain of dependent load rounds (ceil(nsplit / kGroup) of
// them), so requests split many ways take a wider group and more CTAs per
// row block: kParts = 4 gives a CTA 16 chunks (8 warps, two chunks each),
// kParts = 16 gives it 4 (4 warps, one chunk each).
template <int kParts>
__host__ __device__ constexpr int comb_threads() { return kParts == 4 ? 256 : 32 * (kChunks / kParts); }
// column split of a launch whose widest job has more than 8 splits
constexpr int kWideParts = 16;
template <int kGroup, int kParts>
__device__ __forceinline__ void combine_body(const CombineJob job, const DecodeArgs& a, int row_block, int part) {
  static_assert(kParts == 4 || kParts == 16 || kParts == 32 || kParts == 64, "column split");
  constexpr int kCtaChunks = kChunks / kParts;
  constexpr int kWarps = comb_threads<kParts>() / 32;
  constexpr int kPerWarp = kCtaChunks / kWarps;  // a warp's chunks: c0 + warp + kWarps * k
  extern __shared__ float s_w[];  // [nsplit][32] weights (0 for -inf splits)
  const int M = a.rows;  // partial-row stride: the planned rows per request
  const int r0 = row_block * kCombRows;
  const int c0 = part * kCtaChunks;
  // this request's query rows (fewer than M in a ragged batch) and where
  // they go in out / lse
  const int2 q = request_q(a, job.req);
  const int nrows = min(kCombRows, q.y * a.num_heads - r0);
  if (nrows <= 0) return;  // whole CTA: no row of this block belongs to the request
  const size_t orow0 = (size_t)q.x * a.num_heads + r0;
  __shared__ uint4 s_out[kCombRows][kCtaChunks + 1];

  const int r = threadIdx.x & 31;  // row within the block
  const int cw = threadIdx.x >> 5;  // warp
  const uint4* po = reinterpret_cast<const uint4*>(a.part_o) + ((size_t)job.slot_begin * kChunks + c0 + cw) * M + r0 + r;
  const size_t split_stride = (size_t)kChunks * M;
  // The partials of the first kGroup splits do not depend on the weights:
  // their loads go out before the lse values are even read, so the two
  // memory round trips overlap.
  uint4 v[kGroup][kPerWarp];
#pragma unroll
  for (int g = 0; g < kGroup; ++g)
#pragma unroll
    for (int k = 0; k < kPerWarp; ++k)
      v[g][k] = (r < nrows && g < job.nsplit) ? __ldg(po + g * split_stride + (size_t)(kWarps * k) * M)
                                              : make_uint4(0, 0, 0, 0);

  if (threadIdx.x < kCombRows) {
    // A split with lse = NaN (a NaN score in its keys) makes the row NaN, as
    // in the definition: the maximum propagates NaN (max.NaN), and from it
    // the sum, the lse and every weight.
    float mx = -CUDART_INF_F, tot = 0.f;
    const float* pl = a.part_lse + (size_t)job.slot_begin * M + r0 + r;
    if (r < nrows) {
      for (int s = 0; s < job.nsplit; ++s) mx = max_nan(mx, __ldg(pl + (size_t)s * M));
      if (mx != -CUDART_INF_F)
        for (int s = 0; s < job.nsplit; ++s) tot += __expf(__ldg(pl + (size_t)s * M) - mx);
      if (blockIdx.z == 0) a.lse[orow0 + r] = tot == 0.f ? -CUDART_INF_F : mx + __logf(tot);
    }
    const float inv = tot == 0.f ? 0.f : 1.f / tot;
    for (int s = 0; s < job.nsplit; ++s) {
      const float l = r < nrows ? __ldg(pl + (size_t)s * M) : -CUDART_INF_F;
      s_w[s * kCombRows + r] = (tot == 0.f || l == -CUDART_INF_F) ? 0.f : __expf(l - mx) * inv;
    }
  }
  __syncthreads();

  float acc[kPerWarp][8];
#pragma unroll
  for (int k = 0; k < kPerWarp; ++k)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[k][e] = 0.f;
  if (r < nrows) {
    for (int s0 = 0; s0 < job.nsplit; s0 += kGroup) {
      if (s0 > 0) {
#pragma unroll
        for (int g = 0; g < kGroup; ++g)
#pragma unroll
          for (int k = 0; k < kPerWarp; ++k)
            v[g][k] = s0 + g < job.nsplit ? __ldg(po + (s0 + g) * split_stride + (size_t)(kWarps * k) * M)
                                          : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int g = 0; g < kGroup; ++g) {
        // a split with weight 0 (lse = -inf, or past nsplit) adds nothing;
        // its partial may hold anything, so it is skipped, not multiplied
        const float wgt = s0 + g < job.nsplit ? s_w[(s0 + g) * kCombRows + r] : 0.f;
        if (wgt == 0.f) continue;
#pragma unroll
        for (int k = 0; k < kPerWarp; ++k) {
          const uint32_t w4[4] = {v[g][k].x, v[g][k].y, v[g][k].z, v[g][k].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            acc[k][2 * e] = fmaf(wgt, bf_lo(w4[e]), acc[k][2 * e]);
            acc[k][2 * e + 1] = fmaf(wgt, bf_hi(w4[e]), acc[k][2 * e + 1]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int k = 0; k < kPerWarp; ++k) {
    uint32_t q[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      __nv_bfloat162 h = __floats2bfloat162_rn(acc[k][2 * e], acc[k][2 * e + 1]);
      q[e] = *reinterpret_cast<uint32_t*>(&h);
    }
    s_out[r][cw + kWarps * k] = make_uint4(q[0], q[1], q[2], q[3]);
  }
  __syncthreads();
  // 32 rows x kCtaChunks 16-byte chunks: kCtaChunks consecutive threads write
  // one row segment with contiguous 16-byte stores
  constexpr int kRowsPerPass = comb_threads<kParts>() / kCtaChunks;
  const int lc = threadIdx.x % kCtaChunks;
  for (int rr = threadIdx.x / kCtaChunks; rr < nrows; rr += kRowsPerPass) {
    const size_t row = orow0 + rr;
    uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) + row * kLatent + kChunkCols * c0) + lc;
    *dst = s_out[rr][lc];
  }
}

// Launched as a programmatic dependent of the main kernel: the launch
// overlaps the main kernel's tail; the partials are read after the wait
// (which returns once the main grid has completed and its writes are
// visible; without the launch attribute it returns at once).
template <int CAP, int kGroup, int kParts>
__global__ void __launch_bounds__(comb_threads<kParts>()) combine_kernel(const __grid_constant__ CombineList<CAP> jobs,
                                                                       const __grid_constant__ DecodeArgs a) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  combine_body<kGroup, kParts>(jobs.job[blockIdx.x], a, blockIdx.y, blockIdx.z);
}

// Device plan: the job list is in the workspace, written by the planner
// grid two launches earlier (read at L2, ld.global.cg, like the schedule);
// the grid covers the most jobs any plan for the batch can have and CTAs past
// the actual count return.
__global__ void __launch_bounds__(256) combine_kernel_dev(const CombineList<kJobCap>* jobs,
                                                          const __grid_constant__ DecodeArgs a) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if ((int)blockIdx.x >= __ldcg(&jobs->num_jobs)) return;
  const CombineJob* j = &jobs->job[blockIdx.x];  // 4-byte loads: no alignment assumed
  combine_body<4, 4>(CombineJob{__ldcg(&j->req), __ldcg(&j->slot_begin), __ldcg(&j->nsplit), 0}, a, blockIdx.y,
                     blockIdx.z);
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
  // splits in flight per load round: enough for the widest job, within
  // reason; more than 8 splits: a sixteenth of the row per CTA
  const int parts = maxsplit <= 8 ? 4 : kWideParts;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)jobs.size(), (unsigned)((a.rows + kCombRows - 1) / kCombRows), (unsigned)parts);
  cfg.blockDim = dim3(parts == 4 ? comb_threads<4>() : comb_threads<kWideParts>());
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  // programmatic dependent launch: the grid may start while the main kernel
  // (the previous launch on the stream) finishes; see griddepcontrol.wait
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (maxsplit <= 4) return cudaLaunchKernelEx(&cfg, combine_kernel<CAP, 4, 4>, list, a);
  if (maxsplit <= 8) return cudaLaunchKernelEx(&cfg, combine_kernel<CAP, 8, 4>, list, a);
  return cudaLaunchKernelEx(&cfg, combine_kernel<CAP, 16, kWideParts>, list, a);
}

cudaError_t launch_combine(const std::vector<CombineJob>& jobs, const DecodeArgs& a,
                           cudaStream_t stream) {
  if (jobs.empty()) return cudaSuccess;
  return launch_combine_cap<kJobCap>(jobs, a, stream);
}

cudaError_t launch_combine_dev(int workers, const DecodeArgs& a, const void* workspace, cudaStream_t stream) {
  if (workers < 2) return cudaSuccess;  // one worker never splits a request
  const auto* jobs = reinterpret_cast<const CombineList<kJobCap>*>(static_cast<const char*>(workspace) +
                                                                    kDevJobsOffset);
  cudaLaunchConfig_t cfg = {};
  // at most one job per split request: fewer than the workers, and no more
  // than the requests
  const int max_jobs = workers - 1 < a.batch ? workers - 1 : a.batch;
  cfg.gridDim = dim3((unsigned)max_jobs, (unsigned)((a.rows + kCombRows - 1) / kCombRows),
                     (unsigned)(kChunks / kCombChunks));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = (size_t)workers * kCombRows * sizeof(float);  // a request spans <= W workers
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_kernel_dev, jobs, a);
}

}  // namespace mla
