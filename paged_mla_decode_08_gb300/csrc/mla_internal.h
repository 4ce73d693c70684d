// Internal structures shared by the host launcher and the device kernels.
// Not part of the public ABI (include/mla_decode.h).
#pragma once

#include <stddef.h>
#include <stdint.h>

#include <vector>

namespace mla {

constexpr int kTileTokens = 64;      // KV tokens per main-loop tile
constexpr int kSegOverheadTiles = 3; // planner: per-segment cost, in tiles (measured: about 2.6)
constexpr int kMinSplitTiles = 4;    // planner: shortest piece of a split request
constexpr int kMaxWorkers = 128;     // persistent CTA pairs (<= 256 SMs)
constexpr int kMaxRows = 128;        // num_heads * q_len handled by one CTA
constexpr int kLatent = 512;
constexpr int kRope = 64;
constexpr int kKvDim = 576;

// One run of whole tiles of one request, processed by one worker.
struct Segment {
  int32_t req;
  int32_t tile_begin;
  int32_t tile_end;
  int32_t slot;  // partial-result slot, or -1: write out/lse directly
};

// A split request to merge: its partial slots are [slot_begin, slot_begin + nsplit).
struct CombineJob {
  int32_t req;
  int32_t slot_begin;
  int32_t nsplit;
  int32_t pad;
};

// Schedule passed by value as a kernel parameter (no device copy needed,
// nothing to upload, safe to capture in a CUDA graph).
template <int CAP>
struct Schedule {
  int32_t num_workers;
  int32_t num_segments;
  int32_t worker_seg[kMaxWorkers + 1];  // segments of worker w: [worker_seg[w], worker_seg[w+1])
  Segment seg[CAP];
};
constexpr int kSegCapSmall = 448;
constexpr int kSegCapLarge = 1920;

template <int CAP>
struct CombineList {
  int32_t num_jobs;
  int32_t pad[3];
  CombineJob job[CAP];
};
// Every split request spans at least one worker boundary, so a plan has at
// most kMaxWorkers - 1 combine jobs; one capacity covers all plans.
constexpr int kJobCap = 128;
static_assert(kJobCap >= kMaxWorkers - 1, "combine job capacity");

// Device plans (schedule built on the device from the device lengths): the
// workspace starts with the schedule and the combine-job list, then the
// partials, sized for the most a plan can need (2 (W - 1) split slots).  At
// most batch + W - 1 segments, so the batch is bounded by the capacity.
constexpr size_t align256(size_t x) { return (x + 255) / 256 * 256; }
constexpr size_t kDevSchedOffset = 0;
constexpr size_t kDevJobsOffset = align256(sizeof(Schedule<kSegCapLarge>));
constexpr size_t kDevPartOffset = align256(kDevJobsOffset + sizeof(CombineList<kJobCap>));
constexpr int kDevMaxBatch = kSegCapLarge - (kMaxWorkers - 1);

// Pointers and scalars of one decode call, as the kernels see them.
struct DecodeArgs {
  const void* q_nope;  // bf16 [T, H, 512]
  const void* q_pe;    // bf16 [T, H, 64]
  const void* kv;      // bf16 | e4m3 [P, page, 576]
  const int32_t* block_table;
  const int32_t* seq_lens;
  void* out;           // bf16 [T, H, 512]
  float* lse;          // fp32 [T, H]
  void* part_o;        // bf16 [slot][64 chunks of 8 columns][M] (O / l of one split)
  float* part_lse;     // fp32 [slots, M]
  int64_t num_pages;
  int32_t page_size;
  int32_t kv_dtype;
  int32_t bt_stride;
  int32_t batch;
  int32_t q_len;
  int32_t num_heads;
  int32_t rows;        // M = num_heads * q_len
  float score_scale_log2;  // scale * kf * log2(e): logits in base-2 units
  float out_scale;         // kf (value dequantisation)
  const int32_t* cu_q;     // ragged batches: int32 [batch + 1] first query token of each
                           // request (q_len is then the planned maximum); nullptr: uniform
  int32_t num_tokens;      // rows of q_nope / q_pe / out / lse
  int32_t q_e4m3;          // q_nope is the merged e4m3 query [T, H, 576] (q_pe unused)
};

#ifdef __CUDACC__
// First query token and query-token count of request b: (b * q_len, q_len)
// for a uniform batch; (cu_q[b], cu_q[b+1] - cu_q[b]) for a ragged one.  A
// ragged entry outside 0 <= cu_q[b] <= cu_q[b+1] <= num_tokens, or with more
// tokens than the planned maximum, counts as no query token (*bad is set),
// so no access leaves the query and output arrays.
__device__ __forceinline__ int2 request_q(const DecodeArgs& a, int b, bool* bad = nullptr) {
  if (a.cu_q == nullptr) return make_int2(b * a.q_len, a.q_len);
  const int t0 = __ldg(a.cu_q + b), t1 = __ldg(a.cu_q + b + 1);
  if (t0 < 0 || t1 < t0 || t1 > a.num_tokens || t1 - t0 > a.q_len) {
    if (bad) *bad = true;
    return make_int2(0, 0);
  }
  return make_int2(t0, t1 - t0);
}
#endif

}  // namespace mla

// The plan object behind the opaque C handle.
struct mla_plan {
  int batch = 0, page_size = 0, num_heads = 0, q_len = 0, rows = 0;
  bool ragged = false;  // planned from per-request query counts (q_len = their maximum)
  bool device = false;  // schedule built on the device at each decode (segs / jobs empty here)
  int num_sms = 0, num_workers = 0;
  int max_pages = 0;  // ceil(max seq_len / page_size)
  int num_slots = 0;
  size_t ws_bytes = 0, ws_lse_offset = 0;
  size_t ws_part_offset = 0;  // partial outputs (after the schedule area of a device plan)
  int64_t plan_capacity = 0;  // per-worker cost bound the schedule was made with
  std::vector<int32_t> seq_lens;
  std::vector<int32_t> seg_worker;  // worker of each segment (inspection)
  std::vector<mla::Segment> segs;
  std::vector<int32_t> worker_seg;  // [num_workers + 1]
  std::vector<mla::CombineJob> jobs;
};

namespace mla {
// Host planner (mla_plan.cpp).  Returns 0 or an MLA_ERR_* code; on error
// *msg points to a static description.
int build_plan(const int32_t* seq_lens, int batch, int page_size, int num_heads, int q_len,
               int num_sms, mla_plan* plan, const char** msg);
// Device plan: workers and workspace layout only (mla_plan.cpp).
int build_device_plan(int batch, int page_size, int num_heads, int q_len, int num_sms, mla_plan* plan,
                      const char** msg);
}  // namespace mla
