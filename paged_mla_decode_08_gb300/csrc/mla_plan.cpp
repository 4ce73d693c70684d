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
// OVH = 2 tiles of fixed work (query load, epilogue).  With S segments,
//     total = sum_b n_b + OVH * S,   bound(w) = ceil((w + 1) * total / W),
// worker w is filled until the cumulative cost of everything poured so far
// reaches bound(w).  Requests are walked in order: a request that fits into
// the worker's remaining room goes there whole; otherwise the worker takes
// `room` tiles of it (a worker whose room is below MIN = 4 tiles and that
// already holds work is closed first), and if that would leave fewer than MIN
// tiles behind it takes `left - MIN` instead (or everything when that is
// below MIN).  Because the bounds are absolute, rounding never accumulates.
// The last worker takes whatever is left.  S is not known before pouring:
// the first pass assumes S = B + W - 1, the second uses the first pass's S.  Zero-length requests get
// one empty segment (it writes out = 0, lse = -inf).  A request cut into
// k >= 2 segments gets k consecutive partial slots; a single-segment request
// is written directly.
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
  int64_t nsegs = (int64_t)batch + W - 1;
  for (int pass = 0; pass < 2; ++pass) {
  total = tiles_sum + (int64_t)kSegOverheadTiles * nsegs;
  auto bound = [&](int w) -> int64_t { return ((int64_t)(w + 1) * total + W - 1) / W; };

  p->segs.clear(); p->seg_worker.clear();
  int w = 0;
  bool w_used = false;
  int64_t cum = 0;
  auto advance = [&]() {
    while (w < W - 1 && cum >= bound(w)) { ++w; w_used = false; }
  };
  for (int b = 0; b < batch; ++b) {
    if (tiles[b] == 0) {
      p->segs.push_back(Segment{b, 0, 0, -1});
      p->seg_worker.push_back(w);
      w_used = true;
      cum += kSegOverheadTiles;
      advance();
      continue;
    }
    int64_t t = 0;
    while (t < tiles[b]) {
      const int64_t left = tiles[b] - t;
      const int64_t room = bound(w) - cum - kSegOverheadTiles;
      int64_t n;
      if (w == W - 1 || left <= room) {
        n = left;
      } else if (room < kMinSplitTiles) {
        if (w_used) { ++w; w_used = false; continue; }
        n = std::min<int64_t>(left, kMinSplitTiles);
      } else {
        n = room;
        if (left - n < kMinSplitTiles) n = (left - kMinSplitTiles >= kMinSplitTiles) ? left - kMinSplitTiles : left;
      }
      p->segs.push_back(Segment{b, (int32_t)t, (int32_t)(t + n), -1});
      p->seg_worker.push_back(w);
      w_used = true;
      cum += n + kSegOverheadTiles;
      t += n;
      advance();
    }
  }
  nsegs = (int64_t)p->segs.size();
  }

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

}  // namespace mla
