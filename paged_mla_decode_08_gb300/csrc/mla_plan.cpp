// Host split-KV planner.
//
// Role: what FlashMLA's get_mla_metadata provides to tokenspeed flashmla.py
// (FlashMLABackend._init_decode_metadata): a tile schedule that spreads
// ragged requests over the SMs, and per-request split counts.  The rule
// below is this library's own.
//
// Rule.  Cut every request into 64-token tiles, n_b = ceil(L_b / 64).  There
// are W workers (one per CTA pair, W = num_sms / 2, at most 128).  Each
// segment (a run of tiles of one request on one worker) costs its tiles plus
// OVH = 3 tiles of fixed work (query load, epilogue, pipeline refill: a
// clock64 trace of the kernel puts it at about 2.6 tiles).  For a capacity C,
// fill(C) walks the requests in order and pours them into workers 0, 1, ...:
// a request that fits the worker's room (C - cost so far - OVH) goes there
// whole; otherwise, when room >= MIN (= 4) and at least 2 MIN tiles are left,
// the worker takes min(room, left - MIN) tiles (no piece, the rest included,
// is shorter than MIN); otherwise a worker that already holds work is closed,
// and an empty one takes MIN tiles (all of them when fewer than 2 MIN are
// left).  The last worker takes whatever is left.  C is the smallest capacity
// (binary search upward from ceil((sum_b n_b + OVH B) / W)) whose fill keeps
// the last worker within C, so the most loaded worker carries about the mean
// cost; the schedule is fill(C).  A zero-length request gets one empty
// segment (it writes out = 0, lse = -inf), placed on the next worker when it
// does not fit.  A request cut into k >= 2 segments gets k consecutive
// partial slots; a single-segment request is written directly.
#include <algorithm>
#include <cstdint>

#include "../../include/mla_decode.h"
#include "mla_internal.h"

namespace mla {

int build_plan(const int32_t* seq_lens, int batch, int page_size, int num_heads, int q_len,
               int num_sms, mla_plan* p, const char** msg) {
  if (seq_lens == nullptr) { *msg = "seq_lens_host is NULL"; return MLA_ERR_ARG; }
  if (batch < 1) { *msg = "batch must be >= 1"; return MLA_ERR_ARG; }
  if (page_size != 32 && page_size != 64) { *msg = "page_size must be 32 or 64"; return MLA_ERR_ARG; }
  if (num_heads < 1 || q_len < 1) { *msg = "num_heads and q_len must be >= 1"; return MLA_ERR_ARG; }
  if ((int64_t)num_heads * q_len > kMaxRows) {
    *msg = "num_heads * q_len must be <= 128";
    return MLA_ERR_ARG;
  }
  if (num_sms < 2) { *msg = "num_sms must be >= 2"; return MLA_ERR_ARG; }

  const int W = std::min(num_sms / 2, kMaxWorkers);
  p->batch = batch; p->page_size = page_size; p->num_heads = num_heads; p->q_len = q_len;
  p->rows = num_heads * q_len; p->num_sms = num_sms; p->num_workers = W;
  p->seq_lens.assign(seq_lens, seq_lens + batch);

  std::vector<int64_t> tiles(batch);
  int64_t total = 0;
  int64_t max_len = 0;
  for (int b = 0; b < batch; ++b) {
    if (seq_lens[b] < 0) { *msg = "seq_lens must be >= 0"; return MLA_ERR_ARG; }
    tiles[b] = ((int64_t)seq_lens[b] + kTileTokens - 1) / kTileTokens;
    total += tiles[b] + kSegOverheadTiles;
    max_len = std::max<int64_t>(max_len, seq_lens[b]);
  }
  p->max_pages = (int)((max_len + page_size - 1) / page_size);
  int64_t tiles_sum = total - (int64_t)kSegOverheadTiles * batch;
  (void)tiles_sum;

  // Capacity-bounded greedy fill: workers take requests in order, each up to
  // a cost of `cap` (tiles + kSegOverheadTiles per segment); a request that
  // does not fit is cut at the capacity, with no piece shorter than
  // kMinSplitTiles (a worker that cannot take such a piece moves on; only a
  // worker still empty may overshoot, by less than kMinSplitTiles).  The last
  // worker takes whatever is left.  Returns the last worker's cost.
  auto fill = [&](int64_t cap, bool emit) -> int64_t {
    if (emit) { p->segs.clear(); p->seg_worker.clear(); }
    int w = 0;
    bool used = false;
    int64_t cum = 0;
    auto next_worker = [&]() { ++w; cum = 0; used = false; };
    for (int b = 0; b < batch; ++b) {
      if (tiles[b] == 0) {
        if (used && w < W - 1 && cum + kSegOverheadTiles > cap) next_worker();
        if (emit) { p->segs.push_back(Segment{b, 0, 0, -1}); p->seg_worker.push_back(w); }
        used = true;
        cum += kSegOverheadTiles;
        continue;
      }
      int64_t t = 0;
      while (t < tiles[b]) {
        const int64_t left = tiles[b] - t;
        const int64_t room = cap - cum - kSegOverheadTiles;
        int64_t n;
        if (w == W - 1 || left <= room) {
          n = left;
        } else if (room >= kMinSplitTiles && left - kMinSplitTiles >= kMinSplitTiles) {
          n = std::min(room, left - kMinSplitTiles);  // the rest stays >= kMinSplitTiles
        } else if (used) {
          next_worker();
          continue;
        } else {
          n = std::min(left, (int64_t)kMinSplitTiles);  // an empty worker takes at least a minimum piece
          if (left - n < kMinSplitTiles) n = left;
        }
        if (emit) {
          p->segs.push_back(Segment{b, (int32_t)t, (int32_t)(t + n), -1});
          p->seg_worker.push_back(w);
        }
        used = true;
        cum += n + kSegOverheadTiles;
        t += n;
      }
    }
    return (w == W - 1) ? cum : 0;
  };
  // smallest capacity whose fill leaves the last worker within it
  int64_t lo = 1, hi = 1;
  {
    int64_t sum = 0;
    for (int b = 0; b < batch; ++b) sum += tiles[b] + kSegOverheadTiles;
    lo = std::max<int64_t>(1, (sum + W - 1) / W);
    hi = sum + (int64_t)kSegOverheadTiles * W + kMinSplitTiles;
  }
  while (lo < hi) {
    const int64_t mid = lo + (hi - lo) / 2;
    if (fill(mid, false) <= mid) hi = mid;
    else lo = mid + 1;
  }
  fill(lo, true);
  p->plan_capacity = lo;

  // split counts and partial slots
  std::vector<int> nseg(batch, 0);
  for (const Segment& s : p->segs) nseg[s.req]++;
  std::vector<int> slot_base(batch, -1);
  int slots = 0;
  p->jobs.clear();
  for (int b = 0; b < batch; ++b) {
    if (nseg[b] >= 2) {
      slot_base[b] = slots;
      p->jobs.push_back(CombineJob{b, slots, nseg[b], 0});
      slots += nseg[b];
    }
  }
  std::vector<int> seen(batch, 0);
  for (Segment& s : p->segs) {
    if (slot_base[s.req] >= 0) s.slot = slot_base[s.req] + seen[s.req]++;
  }
  p->num_slots = slots;

  // worker ranges (segments are emitted in worker order)
  p->worker_seg.assign(W + 1, 0);
  for (int i = 0; i < (int)p->segs.size(); ++i) p->worker_seg[p->seg_worker[i] + 1] = i + 1;
  for (int i = 1; i <= W; ++i) p->worker_seg[i] = std::max(p->worker_seg[i], p->worker_seg[i - 1]);

  const size_t o_bytes = (size_t)slots * p->rows * kLatent * 2;  // bf16 partial outputs
  p->ws_lse_offset = (o_bytes + 255) / 256 * 256;
  const size_t l_bytes = (size_t)slots * p->rows * sizeof(float);
  p->ws_bytes = slots ? p->ws_lse_offset + (l_bytes + 255) / 256 * 256 : 0;
  *msg = "";
  return MLA_OK;
}

// A device plan fixes only the batch shape: the schedule itself is built by
// the planner kernel (mla_plan_device.cu) from the device lengths at every
// decode, into the head of the workspace, which is sized for the largest
// schedule any lengths can give (2 (W - 1) split slots).
int build_device_plan(int batch, int page_size, int num_heads, int q_len, int num_sms, mla_plan* p,
                      const char** msg) {
  if (batch < 1 || batch > kDevMaxBatch) { *msg = "batch must be in [1, 1793] for a device plan"; return MLA_ERR_ARG; }
  if (page_size != 32 && page_size != 64) { *msg = "page_size must be 32 or 64"; return MLA_ERR_ARG; }
  if (num_heads < 1 || q_len < 1) { *msg = "num_heads and q_len must be >= 1"; return MLA_ERR_ARG; }
  if ((int64_t)num_heads * q_len > kMaxRows) { *msg = "num_heads * q_len must be <= 128"; return MLA_ERR_ARG; }
  if (num_sms < 2) { *msg = "num_sms must be >= 2"; return MLA_ERR_ARG; }
  const int W = std::min(num_sms / 2, kMaxWorkers);
  p->batch = batch; p->page_size = page_size; p->num_heads = num_heads; p->q_len = q_len;
  p->rows = num_heads * q_len; p->num_sms = num_sms; p->num_workers = W;
  p->device = true;
  p->max_pages = 1;  // lengths are unknown: the decode clamps them to the block-table row
  const int slots = 2 * (W - 1);
  p->num_slots = slots;
  p->ws_part_offset = kDevPartOffset;
  const size_t o_bytes = (size_t)slots * p->rows * kLatent * 2;
  p->ws_lse_offset = kDevPartOffset + (o_bytes + 255) / 256 * 256;
  const size_t l_bytes = (size_t)slots * p->rows * sizeof(float);
  p->ws_bytes = p->ws_lse_offset + (l_bytes + 255) / 256 * 256;
  *msg = "";
  return MLA_OK;
}

}  // namespace mla
