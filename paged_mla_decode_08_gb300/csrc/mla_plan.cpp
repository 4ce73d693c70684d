// Host split-KV planner.
//
// Role: what FlashMLA's get_mla_metadata provides to tokenspeed flashmla.py
// (FlashMLABackend._init_decode_metadata): a tile schedule that spreads
// ragged requests over the SMs, and per-request split counts.  The rule
// below is this library's own.
//
// Rule.  Cut every request into 64-token tiles, n_b = ceil(L_b / 64).  There
// are W workers (one per CTA pair, W = num_sms / 2).  Each segment (a run of
// tiles of one request on one worker) costs its tiles plus OVH = 2 tiles of
// fixed work (query load, epilogue).  Budget per worker:
//     cap = max(ceil((sum_b n_b + OVH * B) / W), OVH + MIN)
// with MIN = 4.  Requests are walked in order and poured into workers in
// order: a worker takes as many tiles of the current request as fit into its
// remaining budget (at least MIN), a piece of fewer than MIN tiles is never
// left behind (it stays on the current worker), and a worker whose remaining
// room cannot hold min(left, MIN) tiles is closed.  The last worker takes
// whatever is left.  Zero-length requests get one empty segment (it writes
// out = 0, lse = -inf).  A request cut into k >= 2 segments gets k
// consecutive partial slots; a single-segment request is written directly.
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
  const int64_t cap = std::max<int64_t>((total + W - 1) / W, kSegOverheadTiles + kMinSplitTiles);

  p->segs.clear(); p->seg_worker.clear();
  int w = 0;
  int64_t used = 0;
  auto close_if_full = [&]() {
    if (used >= cap && w < W - 1) { ++w; used = 0; }
  };
  for (int b = 0; b < batch; ++b) {
    if (tiles[b] == 0) {
      p->segs.push_back(Segment{b, 0, 0, -1});
      p->seg_worker.push_back(w);
      used += kSegOverheadTiles;
      close_if_full();
      continue;
    }
    int64_t t = 0;
    while (t < tiles[b]) {
      const int64_t left = tiles[b] - t;
      const int64_t room = cap - used - kSegOverheadTiles;
      if (w < W - 1 && used > 0 && room < std::min<int64_t>(left, kMinSplitTiles)) {
        ++w; used = 0;
        continue;
      }
      int64_t n = (w == W - 1) ? left : std::min(left, std::max<int64_t>(room, kMinSplitTiles));
      if (left - n < kMinSplitTiles) n = left;
      p->segs.push_back(Segment{b, (int32_t)t, (int32_t)(t + n), -1});
      p->seg_worker.push_back(w);
      used += kSegOverheadTiles + n;
      t += n;
      close_if_full();
    }
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

  const size_t o_bytes = (size_t)slots * p->rows * kLatent * sizeof(float);
  p->ws_lse_offset = (o_bytes + 255) / 256 * 256;
  const size_t l_bytes = (size_t)slots * p->rows * sizeof(float);
  p->ws_bytes = slots ? p->ws_lse_offset + (l_bytes + 255) / 256 * 256 : 0;
  *msg = "";
  return MLA_OK;
}

}  // namespace mla
