// Device-side split-KV planner: builds the schedule and the combine-job list
// from the device seq_lens, so that a decode captured once in a CUDA graph
// can be replayed for any lengths with no host round trip (the role of
// FlashMLA's get_mla_metadata in tokenspeed flashmla.py,
// _init_decode_metadata, which runs on the device too).
//
// Rule (restated in tests/test_plan_device.py).  With n_b = ceil(L_b / 64)
// tiles (L_b clamped like the decode does) and cost c_b = n_b + OVH, let P_b
// be the exclusive prefix sum of c_b, C the total and cap = max(ceil(C / W),
// MIN).
// Request b's tiles occupy cost [P_b, P_b + n_b) (its overhead follows
// them); worker w owns cost [w * cap, (w + 1) * cap).  The pieces of b are
// its intersections with the worker intervals, whatever their length: each
// piece pays the segment overhead on its worker, and merging a short piece
// into a neighbour instead would load that neighbour past the capacity (a
// request just longer than cap would land whole on one worker).  A request
// with no tile is one empty segment on the worker holding P_b.
// Requests and their pieces are emitted in order, so segments come out
// sorted by worker.  Split requests (two or more pieces) take consecutive
// partial slots and one combine job each; with every split spanning a worker
// boundary there are at most W - 1 jobs and 2 (W - 1) slots, and at most
// batch + W - 1 segments.
//
// One CTA of as many warps as the batch needs (two requests per thread, up
// to 1024 threads): a single warp for up to 64 requests, whose scans then
// need no block barrier work.  Prefix sums are block scans (one for the
// costs, one for the segment, slot and job counts packed into one 64-bit
// word), and worker_seg is a lower bound of each worker in the sorted
// segment-worker array.  The grid is launched ahead of the decode on the same
// stream and lets the decode's prologue start early (programmatic dependent
// launch).  (Running this rule inside the decode's own prologue instead, in
// every CTA, was measured slower: its cold length load and scans then sit on
// every CTA's path, where here they overlap the decode's launch.)
#include <cuda_runtime.h>
#include <stdint.h>

#include "mla_internal.h"

namespace mla {
namespace devplan {

constexpr int kThreads = 1024;
constexpr int kPerThread = 2;

// Exclusive prefix sum over the block of one 64-bit value per thread; every
// thread also receives the total.
__device__ long long block_exclusive_scan(long long v, long long* total, long long* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    long long w = lane < nwarps ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    s_warp[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const long long before = (warp > 0 ? s_warp[warp - 1] : 0) + x - v;
  *total = s_warp[nwarps - 1];
  __syncthreads();  // s_warp is reused by the next scan
  return before;
}

struct Piece {
  int w0;     // worker of the first piece
  int nseg;   // pieces (>= 1)
};

// Pieces of a request whose tiles occupy cost [p, p + n) (n > 0).
__device__ __forceinline__ Piece pieces_of(long long p, int n, long long cap, int workers) {
  long long w0 = p / cap, w1 = (p + n - 1) / cap;
  if (w1 > workers - 1) w1 = workers - 1;
  if (w0 > w1) w0 = w1;
  return Piece{(int)w0, (int)(w1 - w0 + 1)};
}

__global__ void __launch_bounds__(kThreads, 1)
    plan_kernel(const int32_t* __restrict__ seq_lens, int batch, int cap_tokens, int workers,
                Schedule<kSegCapLarge>* __restrict__ sched, CombineList<kJobCap>* __restrict__ jobs) {
  // the decode (launched next, as a programmatic dependent) may set up its
  // shared memory and TMEM while this grid runs; it reads the schedule only
  // after this grid completed
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ long long s_warp[32];
  __shared__ int16_t s_seg_worker[kSegCapLarge];

  // ---- per-request tiles and cost, prefix sums
  int n[kPerThread];
  long long cost = 0;
#pragma unroll
  for (int k = 0; k < kPerThread; ++k) {
    const int b = threadIdx.x * kPerThread + k;
    int L = b < batch ? __ldg(seq_lens + b) : 0;
    L = L < 0 ? 0 : (L < cap_tokens ? L : cap_tokens);  // the decode's clamp
    n[k] = (L + kTileTokens - 1) / kTileTokens;
    cost += b < batch ? n[k] + kSegOverheadTiles : 0;
  }
  long long total;
  long long p = block_exclusive_scan(cost, &total, s_warp);
  // at least MIN tiles per worker interval
  long long cap = (total + workers - 1) / workers;
  cap = cap < kMinSplitTiles ? kMinSplitTiles : cap;

  Piece pc[kPerThread];
  long long pb[kPerThread];
  int nseg_t = 0, slots_t = 0, jobs_t = 0;
#pragma unroll
  for (int k = 0; k < kPerThread; ++k) {
    const int b = threadIdx.x * kPerThread + k;
    pb[k] = p;
    if (b < batch) {
      if (n[k] == 0) {
        long long w = p / cap;
        pc[k] = Piece{(int)(w < workers - 1 ? w : workers - 1), 1};
      } else {
        pc[k] = pieces_of(p, n[k], cap, workers);
      }
      p += n[k] + kSegOverheadTiles;
      nseg_t += pc[k].nseg;
      if (pc[k].nseg > 1) {
        slots_t += pc[k].nseg;
        ++jobs_t;
      }
    } else {
      pc[k] = Piece{0, 0};
    }
  }
  // one scan for the three counts, 21 bits each (each total is at most
  // batch + workers - 1 < 2^21)
  long long packed_total;
  const long long packed = block_exclusive_scan((long long)nseg_t | ((long long)slots_t << 21) | ((long long)jobs_t << 42),
                                                &packed_total, s_warp);
  const long long m21 = (1LL << 21) - 1;
  int seg_base = (int)(packed & m21);
  int slot_base = (int)((packed >> 21) & m21);
  int job_base = (int)(packed >> 42);
  const long long nseg_total = packed_total & m21, jobs_total = packed_total >> 42;

  // ---- segments and combine jobs
#pragma unroll
  for (int k = 0; k < kPerThread; ++k) {
    const int b = threadIdx.x * kPerThread + k;
    if (b >= batch) continue;
    const int ns = pc[k].nseg;
    for (int i = 0; i < ns; ++i) {
      const int w = pc[k].w0 + i;
      Segment sg;
      sg.req = b;
      sg.tile_begin = i == 0 ? 0 : (int)((long long)w * cap - pb[k]);
      sg.tile_end = i == ns - 1 ? n[k] : (int)((long long)(w + 1) * cap - pb[k]);
      sg.slot = ns > 1 ? slot_base + i : -1;
      sched->seg[seg_base + i] = sg;
      s_seg_worker[seg_base + i] = (int16_t)w;
    }
    if (ns > 1) {
      CombineJob j;
      j.req = b;
      j.slot_begin = slot_base;
      j.nsplit = ns;
      j.pad = 0;
      jobs->job[job_base++] = j;
      slot_base += ns;
    }
    seg_base += ns;
  }
  __syncthreads();

  // ---- worker_seg[w] = first segment whose worker is >= w
  const int total_segs = (int)nseg_total;
  for (int w = threadIdx.x; w <= workers; w += blockDim.x) {
    int lo = 0, hi = total_segs;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (s_seg_worker[mid] < w) lo = mid + 1;
      else hi = mid;
    }
    sched->worker_seg[w] = lo;
  }
  if (threadIdx.x == 0) {
    sched->num_workers = workers;
    sched->num_segments = total_segs;
    jobs->num_jobs = (int)jobs_total;
  }
}

}  // namespace devplan

cudaError_t launch_plan_device(const int32_t* seq_lens, int batch, int cap_tokens, int workers, void* workspace,
                               cudaStream_t stream) {
  auto* sched = reinterpret_cast<Schedule<kSegCapLarge>*>(static_cast<char*>(workspace) + kDevSchedOffset);
  auto* jobs = reinterpret_cast<CombineList<kJobCap>*>(static_cast<char*>(workspace) + kDevJobsOffset);
  // two requests per thread, whole warps, at most kThreads
  int threads = ((batch + devplan::kPerThread - 1) / devplan::kPerThread + 31) / 32 * 32;
  threads = threads < 32 ? 32 : (threads > devplan::kThreads ? devplan::kThreads : threads);
  devplan::plan_kernel<<<1, threads, 0, stream>>>(seq_lens, batch, cap_tokens, workers, sched, jobs);
  return cudaGetLastError();
}

}  // namespace mla
