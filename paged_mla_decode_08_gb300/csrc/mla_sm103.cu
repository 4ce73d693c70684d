// Split-KV paged MLA decode main kernel for sm_103a: TMA page gathers,
// tcgen05 MMAs with TMEM accumulators, online softmax in registers.
//
// Work decomposition.  One persistent CTA pair (a 2-CTA cluster) per
// worker of the host schedule walks that worker's segments (runs of 64-token
// tiles of one request).  The two CTAs split the 512 latent columns: CTA r
// owns c_kv columns [256r, 256r+256) and rope columns [32r, 32r+32), so each
// reads exactly half of every cache row from HBM and nothing twice.
//   S_r = Q[:, half r] . KV[:, half r]^T    (M = 128 query rows, N = 64 keys,
//                                           K = 256 + 32)      -> TMEM
//   S   = S_0 + S_1                         (partial scores swapped through
//                                           distributed shared memory as
//                                           24-bit codes, see score24)
//   P   = exp2(S * scale*log2e - m)         (both CTAs compute the same P)
//   O_r += P . c_kv[:, half r]              (M = 128, N = 256, K = 64) -> TMEM
// The cache tile in shared memory serves both products: K-major as the B
// operand of S, MN-major as the B operand of P.V.  The 128 query rows
// (heads x q_len, zero-padded) are the M dimension of every MMA.
//
// TMEM (512 columns): O [0,256), S double buffer [256,320) / [320,384), Q
// latent half [384,512).  Shared memory: 4-stage cache-tile ring (36 KB per
// stage), the rope half of Q (8 KB), the P tile (16 KB, the A operand of
// P.V), a 3-slot ring of half-tile score-exchange buffers (12 KB each)
// written by the peer CTA.
//
// Warp roles (512 threads): warp 0 TMA producer, warp 1 TMEM allocator and
// MMA issuer (S products; with a bf16 cache warp 3 issues the P.V products),
// warps 4-11 softmax / correction / epilogue (two warps per query row block =
// TMEM lane quadrant, each owning half of a tile's keys and half of the
// output columns), warps 12-15 score exchange with the peer CTA, warps 2-3
// e4m3 -> fp16 converters (float8 cache only).  Every wait is
// bounded: on timeout the kernel records an error code in device memory,
// stops every role, waits for its own copies and MMAs, frees TMEM and
// returns.  The one hardware barrier, a quadrant's named barrier for the
// per-tile row maxima, is released by a softmax warp that leaves early: it
// arrives twice, enough for the furthest its partner can get before it
// sees the abort.
//
// Float8 (e4m3) cache.  The same kernel, instantiated with F8 = true: TMA
// brings raw e4m3 tiles (half the bytes) into a 2-stage fp8 ring, the two
// converter warps expand each tile into one of 3 fp16 operand stages laid
// out like a bf16 stage (cvt.rn.f16x2.e4m3x2 is exact; the two rings share
// the bytes of the bf16 ring), and the MMAs run on fp16
// operands (the query is converted to fp16 once per segment, P is packed
// to fp16).  The per-tensor scale k_scale multiplies the scores and the
// output (it is folded into the score scale and the epilogue scale).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math_constants.h>

#include <mutex>

#include "../../include/mla_decode.h"
#include "mla_internal.h"
#include "sm103_ptx.cuh"

namespace mla {
namespace sm103 {

using namespace mla::ptx;

constexpr int kThreads = 512;  // warps 0-3: producer, MMA, 2 converter (e4m3); 4-11: softmax; 12-15: exchange
constexpr int kStages = 4;  // cache-tile ring stages (bf16); the e4m3 split of the same bytes is below
constexpr int kLatBox = 64 * 128;           // 64 tokens x 64 bf16 columns, 128B swizzle
constexpr int kRopeBox = 64 * 64;           // 64 tokens x 32 bf16 columns, 64B swizzle
constexpr int kStageBytes = 4 * kLatBox + kRopeBox;  // 36864
constexpr int kStageTx = kStageBytes;       // bytes TMA delivers per tile
constexpr int OFF_KV = 0;
// e4m3 cache: the first 144 KB hold kF8OpStages fp16 operand stages (same
// layout as a bf16 stage) followed by kF8Stages fp8 staging stages, each 64
// keys x (256 latent + 32 rope) bytes, unswizzled.  An operand stage is held
// from conversion until its P.V completes, so operand stages are the scarce
// ones; a raw tile is held only from its load until converted.
constexpr int kF8OpStages = 3;
constexpr int kF8Stages = 2;
constexpr int kF8StageBytes = 64 * 288;
constexpr int kF8RopeOff = 64 * 256;
constexpr int OFF_F8 = kF8OpStages * kStageBytes;
static_assert(OFF_F8 + kF8Stages * kF8StageBytes <= kStages * kStageBytes, "fp8 ring fits the operand ring");
template <bool F8>
__host__ __device__ constexpr int op_stages() { return F8 ? kF8OpStages : kStages; }
constexpr int OFF_QROPE = kStages * kStageBytes;       // 128 rows x 64 B
constexpr int OFF_P = OFF_QROPE + 128 * 64;            // P (128 rows x 64 keys bf16, 128B swizzle)
constexpr int kPBytes = 128 * 128;
// Score exchange: a ring of 3 slots, each holding the peer's partial scores
// of one half tile (32 keys) for 128 rows, [16-byte chunk][row], as 24-bit
// codes (see score24).
constexpr int kSlots = 3;
constexpr int OFF_XCHG = OFF_P + kPBytes;
constexpr int kXchgRowBytes = 32 * 3;  // 32 scores of 24 bits: six 16-byte chunks per row
constexpr int kXchgChunks = kXchgRowBytes / 16;
constexpr int kSlotBytes = 128 * kXchgRowBytes;
constexpr int OFF_RED = OFF_XCHG + kSlots * kSlotBytes;  // row max / row sum exchange, 4 KB
constexpr int OFF_SINK = OFF_RED + 4 * 2 * 128 * 4;      // per slot 128 words: the peer's "read done" notes
constexpr int kNoteBytes = 128 * 4;
constexpr int OFF_SEGLEN = OFF_SINK + kSlots * kNoteBytes;  // key counts of the worker's first segments
constexpr int kSegLenCache = 64;
constexpr int OFF_SEGQ = OFF_SEGLEN + kSegLenCache * 4;     // ... and their (first token, query count)
constexpr int OFF_SEGS = OFF_SEGQ + kSegLenCache * 8;       // device plan: the segments themselves
constexpr int OFF_BAR = OFF_SEGS + kSegLenCache * 16;
enum Bar : int {
  B_KV_FULL = 0, B_KV_EMPTY = B_KV_FULL + kStages, B_S_FULL = B_KV_EMPTY + kStages, B_P_FULL = B_S_FULL + 2,
  B_PV_DONE, B_Q_READY, B_X_FULL, B_X_EMPTY = B_X_FULL + kSlots, B_TAIL = B_X_EMPTY + kSlots, B_FINAL,
  B_PAIR_L,                   // [quad]: the two warps of a quadrant swap row sums at a segment's end
                              // (their per-tile row maxima go through named barriers 1-4)
  B_S_LOADED = B_PAIR_L + 4,  // [tile parity]: exchange warps hold S in registers
  B_S_FREE = B_S_LOADED + 2,  // [tile parity]: softmax warps too; the S buffer may take the next S
  B_F8_FULL = B_S_FREE + 2,   // [fp8 stage]: TMA delivered the raw e4m3 tile
  B_F8_EMPTY = B_F8_FULL + kStages,  // [fp8 stage]: converted, may be refilled
  B_FINAL2 = B_F8_EMPTY + kStages,  // the P.V issuer's own drain (two-issuer role split)
  B_COUNT = B_FINAL2 + 1
};
constexpr int OFF_TMEM_SLOT = OFF_BAR + B_COUNT * 8;
constexpr int OFF_ABORT = OFF_TMEM_SLOT + 4;
constexpr int kSmemUsed = OFF_ABORT + 4;
constexpr int kSmemBytes = kSmemUsed + 1024;  // + alignment slack

constexpr uint32_t TM_O = 0, TM_S = 256, TM_Q = 384, kTmemCols = 512;
// bf16 cache: bf16 operands; e4m3 cache: fp16 operands (e4m3 -> fp16 is exact)
template <bool F8>
__host__ __device__ constexpr uint32_t idesc_s() { return idesc_f32acc(128, 64, 0, 0, F8 ? 0u : 1u); }
template <bool F8>
__host__ __device__ constexpr uint32_t idesc_pv() { return idesc_f32acc(128, 256, 0, 1, F8 ? 0u : 1u); }
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P stays <= 256
constexpr long long kTimeoutCycles = 2000000000LL;

static_assert(kSmemBytes <= 232448, "shared memory budget");

__device__ int g_kernel_error;

struct Ctx {
  uint8_t* smem;     // 1024-aligned base
  uint32_t sbase;    // its shared-window address
  volatile int* abort_flag;
  const int* seg_len;  // request_len() of segments seg0 .. seg0 + kSegLenCache - 1
  const int2* seg_q;   // request_q() of the same segments
  int seg0;
  __device__ uint32_t bar(int i) const { return sbase + OFF_BAR + 8 * i; }
};

// Read access to the schedule.  ParamSched: the host plan's schedule, a
// kernel parameter.  GlobalSched: a device plan's schedule in the workspace,
// written by the planner grid while this grid may already be resident, so it
// is read at L2 (ld.global.cg: never from a possibly stale L1 / read-only
// cache line) and only after the grid dependency wait; every CTA of a pair
// then sees the same segments.
template <int CAP>
struct ParamSched {
  const Schedule<CAP>& s;
  __device__ __forceinline__ const void* raw() const { return &s; }
  __device__ __forceinline__ int num_workers() const { return s.num_workers; }
  __device__ __forceinline__ int begin(int w) const { return s.worker_seg[w]; }
  __device__ __forceinline__ int end(int w) const { return s.worker_seg[w + 1]; }
  __device__ __forceinline__ Segment seg(int i) const { return s.seg[i]; }
};
struct GlobalSched {
  const Schedule<kSegCapLarge>* s;
  __device__ __forceinline__ const void* raw() const { return s; }
  __device__ __forceinline__ int num_workers() const { return __ldcg(&s->num_workers); }
  __device__ __forceinline__ int begin(int w) const { return __ldcg(&s->worker_seg[w]); }
  __device__ __forceinline__ int end(int w) const { return __ldcg(&s->worker_seg[w + 1]); }
  // four 4-byte loads: the segment array is only 4-byte aligned (it follows
  // the 4-byte header fields), so no vector load may touch it
  __device__ __forceinline__ Segment seg(int i) const {
    const Segment* p = &s->seg[i];
    return Segment{__ldcg(&p->req), __ldcg(&p->tile_begin), __ldcg(&p->tile_end), __ldcg(&p->slot)};
  }
};

// A device plan's schedule once the prologue has copied this worker's first
// kSegLenCache segments into shared memory: the roles read those like the
// host plan's kernel parameter (no L2 round trip at a segment switch);
// segments past them are read at L2.  begin/end answer for this CTA's own
// worker only.
struct CachedSched {
  const Schedule<kSegCapLarge>* s;
  const Segment* cache;  // shared memory: segments first .. first + cached - 1
  int first, last, cached, workers;
  __device__ __forceinline__ int num_workers() const { return workers; }
  __device__ __forceinline__ int begin(int) const { return first; }
  __device__ __forceinline__ int end(int) const { return last; }
  __device__ __forceinline__ Segment seg(int i) const {
    if (i - first < cached) return cache[i - first];
    const Segment* p = &s->seg[i];
    return Segment{__ldcg(&p->req), __ldcg(&p->tile_begin), __ldcg(&p->tile_end), __ldcg(&p->slot)};
  }
};

// Bounded barrier wait.  false: gave up (timeout here or elsewhere in the CTA).
template <bool kCluster>
__device__ __forceinline__ bool wait_bar(const Ctx& c, uint32_t bar, uint32_t parity, int code) {
  if (kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
    if (*c.abort_flag) return false;
    if (clock64() - t0 > kTimeoutCycles) {
      *c.abort_flag = 1;
      atomicCAS(&g_kernel_error, 0, code);
      return false;
    }
  }
}

// Warp-uniform variant: every lane waits; the warp proceeds only if all did
// (so warp-collective tcgen05 ops never run with part of a warp).
template <bool kCluster>
__device__ __forceinline__ bool wait_bar_warp(const Ctx& c, uint32_t bar, uint32_t parity, int code) {
  const bool ok = wait_bar<kCluster>(c, bar, parity, code);
  return __all_sync(0xffffffffu, ok);
}

// Keys of request b that this launch may visit: the device length, never past
// the block-table row.
__device__ __forceinline__ int request_len(const DecodeArgs& a, int b) {
  int L = a.seq_lens[b];
  L = L < 0 ? 0 : L;
  const int cap = a.bt_stride * a.page_size;
  return L < cap ? L : cap;
}

// request_len() of schedule segment s, from the copy every CTA takes at start
// (one memory round trip for all its segments instead of one per segment
// switch in every role)
template <class S>
__device__ __forceinline__ int seg_len(const Ctx& c, const S& sched, const DecodeArgs& a, int s) {
  const int k = s - c.seg0;
  return k < kSegLenCache ? c.seg_len[k] : request_len(a, sched.seg(s).req);
}

// request_q() with a malformed ragged entry recorded in the error word
__device__ __forceinline__ int2 request_q_checked(const DecodeArgs& a, int b) {
  bool bad = false;
  const int2 q = request_q(a, b, &bad);
  if (bad) atomicCAS(&g_kernel_error, 0, 0x501);
  return q;
}

// (first query token, query count) of schedule segment s, cached like seg_len
template <class S>
__device__ __forceinline__ int2 seg_q(const Ctx& c, const S& sched, const DecodeArgs& a, int s) {
  const int k = s - c.seg0;
  return k < kSegLenCache ? c.seg_q[k] : request_q_checked(a, sched.seg(s).req);
}

// Row of out / lse that query row `row` of a request with (first token,
// query count) q writes, or -1 when the request has fewer rows.
__device__ __forceinline__ int out_row(int2 q, int num_heads, int row) {
  return row < q.y * num_heads ? q.x * num_heads + row : -1;
}

__device__ __forceinline__ int segment_tiles(const Segment& sg, int L) {
  const int last = (L + kTileTokens - 1) / kTileTokens;
  const int e = sg.tile_end < last ? sg.tile_end : last;
  return e > sg.tile_begin ? e - sg.tile_begin : 0;
}

// ------------------------------------------------------------------ producer

template <class S, bool F8, bool Q8>
__device__ void producer(const Ctx& c, const S& sched, const DecodeArgs& a, const CUtensorMap* tm_lat,
                         const CUtensorMap* tm_rope, int worker, int rank) {
  const int lane = threadIdx.x & 31;
  const int oob_row = (int)(a.num_pages * a.page_size);  // first row past the pool: zero-filled by TMA
  const int pieces = kTileTokens / a.page_size;           // pages per tile: 1 or 2
  int j = 0, tails = 0;
  bool ok = true;
  for (int s = sched.begin(worker); ok && s < sched.end(worker); ++s) {
    const Segment sg = sched.seg(s);
    const int L = seg_len(c, sched, a, s);
    const int nt = segment_tiles(sg, L);
    const int32_t* bt = a.block_table + (size_t)sg.req * a.bt_stride;
    // block-table entries of the segment's pages, 32 per load (one per
    // lane), the next 32 requested while the current ones are used: page
    // lookups add no memory latency per tile.  Entries past the request's
    // length are read (inside the row) but never used.
    const int pg_begin = sg.tile_begin * pieces;
    const int pg_end = min(sg.tile_end * pieces, a.bt_stride);
    auto load_chunk = [&](int ch) {
      const int q = pg_begin + (ch << 5) + lane;
      return q < pg_end ? __ldg(bt + q) : -1;
    };
    int chunk = 0, pid_cur = load_chunk(0), pid_next = load_chunk(1);
    auto page_id = [&](int pg) {  // warp-uniform pg >= the previous one
      const int ch = (pg - pg_begin) >> 5;
      while (chunk < ch) {
        pid_cur = pid_next;
        pid_next = load_chunk(++chunk + 1);
      }
      return __shfl_sync(0xffffffffu, pid_cur, (pg - pg_begin) & 31);
    };
    if (nt > 0 && lane == 0) {
      // the exchange warps load this request's query when the segment
      // starts: pull it into L2 now, a few tiles ahead (its rows are
      // contiguous; 16-byte multiples)
      const int2 q = seg_q(c, sched, a, s);
      const size_t r0 = (size_t)q.x * a.num_heads;
      const uint32_t nr = (uint32_t)(q.y * a.num_heads);
      if (nr > 0 && Q8) {
        prefetch_l2_bulk(static_cast<const uint8_t*>(a.q_nope) + r0 * kKvDim, nr * kKvDim);  // merged e4m3 rows
      } else if (nr > 0) {
        prefetch_l2_bulk(reinterpret_cast<const __nv_bfloat16*>(a.q_nope) + r0 * kLatent, nr * kLatent * 2);
        prefetch_l2_bulk(reinterpret_cast<const __nv_bfloat16*>(a.q_pe) + r0 * kRope, nr * kRope * 2);
      }
    }
    for (int jj = 0; jj < nt; ++jj, ++j) {
      const int stage = j % (F8 ? kF8Stages : kStages);
      if (F8) {
        // raw e4m3 tile into the fp8 ring; the converter warps expand it
        if (j >= kF8Stages && !wait_bar_warp<false>(c, c.bar(B_F8_EMPTY + stage), ((j / kF8Stages) - 1) & 1, 0x103)) {
          ok = false;
          break;
        }
        const int tok0 = (sg.tile_begin + jj) * kTileTokens;
        const int pid0 = page_id((sg.tile_begin + jj) * pieces);
        const int pid1 = pieces > 1 ? page_id((sg.tile_begin + jj) * pieces + 1) : -1;
        if (lane == 0) {
          const uint64_t pol = policy_evict_first();  // see the bf16 copies below
          const uint32_t full = c.bar(B_F8_FULL + stage);
          const uint32_t dst = c.sbase + OFF_F8 + stage * kF8StageBytes;
          mbar_arrive_expect_tx(full, kF8StageBytes);
          for (int pc = 0; pc < pieces; ++pc) {
            const int ptok = tok0 + pc * a.page_size;
            int y = oob_row;
            if (ptok < L) {
              const int pid = pc ? pid1 : pid0;
              if (pid >= 0 && pid < a.num_pages) y = pid * a.page_size;
            }
            const uint32_t rows = pc * a.page_size;
            tma_load_2d_hint(dst + rows * 256, tm_lat, full, 256 * rank, y, pol);
            tma_load_2d_hint(dst + kF8RopeOff + rows * 32, tm_rope, full, 512 + 32 * rank, y, pol);
          }
        }
        __syncwarp();
        continue;
      }
      // The first fill of the ring goes out one tile at a time, each tile
      // once the previous one has landed.  At kernel start every CTA's copies
      // compete for HBM; a first tile that travels alone starts the score /
      // softmax chain microseconds earlier than one that shares the wire
      // with the whole fill, and the later tiles arrive while the chain
      // works on it.
      if (j >= 1 && j < kStages && !wait_bar_warp<false>(c, c.bar(B_KV_FULL + (j - 1)), 0, 0x104)) {
        ok = false;
        break;
      }
      if (j >= kStages && !wait_bar_warp<false>(c, c.bar(B_KV_EMPTY + stage), ((j / kStages) - 1) & 1, 0x101)) {
        ok = false;
        break;
      }
      const int t = sg.tile_begin + jj;
      const int tok0 = t * kTileTokens;
      const bool tail = tok0 + kTileTokens > L;
      const uint32_t full = c.bar(B_KV_FULL + stage);
      const uint32_t land = tail ? c.bar(B_TAIL) : full;
      const uint32_t dst = c.sbase + OFF_KV + stage * kStageBytes;
      const int pid0 = page_id(t * pieces);
      const int pid1 = pieces > 1 ? page_id(t * pieces + 1) : -1;
      if (lane == 0) {
        // every cache tile is read once per decode: an evict-first L2 policy
        // keeps the stream from displacing what is read again (queries,
        // block tables, the partials the combine reads next) or what other
        // kernels left dirty there (measured: 3-4 % off the main kernel on
        // the 64- and 8-request bf16 batches after an L2 flush)
        const uint64_t pol = policy_evict_first();
        mbar_arrive_expect_tx(land, kStageTx);
        for (int pc = 0; pc < pieces; ++pc) {
          const int ptok = tok0 + pc * a.page_size;
          int y = oob_row;
          if (ptok < L) {
            const int pid = pc ? pid1 : pid0;
            if (pid >= 0 && pid < a.num_pages) y = pid * a.page_size;
          }
          const uint32_t rows = pc * a.page_size;
#pragma unroll
          for (int bx = 0; bx < 4; ++bx)
            tma_load_2d_hint(dst + bx * kLatBox + rows * 128, tm_lat, land, 256 * rank + 64 * bx, y, pol);
          tma_load_2d_hint(dst + 4 * kLatBox + rows * 64, tm_rope, land, 512 + 32 * rank, y, pol);
        }
      }
      __syncwarp();
      if (tail) {
        // rows past the request's length hold whatever the cache holds there:
        // zero them so 0-probability keys cannot inject NaN/Inf into P.V
        if (!wait_bar_warp<false>(c, land, tails & 1, 0x102)) { ok = false; break; }
        ++tails;
        const int r0 = L - tok0;  // first dead row, 1..63
        uint8_t* st = c.smem + OFF_KV + stage * kStageBytes;
        for (int r = r0 + (lane >> 3); r < kTileTokens; r += 4) {
          const int ch = lane & 7;  // 16-byte chunk of the row
#pragma unroll
          for (int bx = 0; bx < 4; ++bx)
            *reinterpret_cast<uint4*>(st + bx * kLatBox + r * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
          if (ch < 4) *reinterpret_cast<uint4*>(st + 4 * kLatBox + r * 64 + ch * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(full);
      }
    }
  }
  // drain: the copies of the last stages must have landed before the CTA leaves
  const int issued = j;
  const int landed_bar = F8 ? B_F8_FULL : B_KV_FULL;
  constexpr int ring = F8 ? kF8Stages : kStages;
  for (int k = issued - 1; k >= 0 && k >= issued - ring; --k) {
    const long long t0 = clock64();
    while (!mbar_try_wait(c.bar(landed_bar + (k % ring)), (k / ring) & 1) && clock64() - t0 < kTimeoutCycles) {
    }
  }
}

// ------------------------------------------------------------------ e4m3 converter

// Warps 2-3 (e4m3 cache only): expand each raw tile of the fp8 ring into an
// fp16 operand stage laid out exactly like a bf16 stage (K-major 128B-swizzled
// latent boxes, 64B-swizzled rope box), with cvt.rn.f16x2.e4m3x2 (exact:
// every e4m3 value is an fp16 value).  Rows past the request's length are
// written as zeros so 0-probability keys cannot inject NaN/Inf into P.V.
// k_scale is not applied here: it is folded into the score scale and the
// output scale.
template <class S>
__device__ void converter(const Ctx& c, const S& sched, const DecodeArgs& a, int worker) {
  const int w = (threadIdx.x >> 5) - 2;  // 0 or 1
  const int lane = threadIdx.x & 31;
  int j = 0;
  bool ok = true;
  for (int s = sched.begin(worker); ok && s < sched.end(worker); ++s) {
    const Segment sg = sched.seg(s);
    const int L = seg_len(c, sched, a, s);
    const int nt = segment_tiles(sg, L);
    for (int jj = 0; jj < nt; ++jj, ++j) {
      const int fs = j % kF8Stages, os = j % kF8OpStages;
      if (!wait_bar_warp<false>(c, c.bar(B_F8_FULL + fs), (j / kF8Stages) & 1, 0x501)) { ok = false; break; }
      if (j >= kF8OpStages &&
          !wait_bar_warp<false>(c, c.bar(B_KV_EMPTY + os), ((j / kF8OpStages) - 1) & 1, 0x502)) {
        ok = false;
        break;
      }
      const int live = min(kTileTokens, L - (sg.tile_begin + jj) * kTileTokens);  // rows < live hold keys
      const uint32_t src = c.sbase + OFF_F8 + fs * kF8StageBytes;
      const uint32_t dst = c.sbase + OFF_KV + os * kStageBytes;
      // latent: a warp converts one row per step, lane = 16-byte output chunk
      // (8 keys' worth of bytes in, contiguous 256 B per warp read); eight
      // rows' loads are issued before the first conversion so their shared
      // memory latency overlaps
      const int bx = lane >> 3, ch = lane & 7;
#pragma unroll 1
      for (int b8 = 0; b8 < kTileTokens / 16; ++b8) {
        uint2 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = 16 * b8 + 2 * i + w;
          v[i] = r < live ? ld_shared_v2(src + r * 256 + lane * 8) : make_uint2(0, 0);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = 16 * b8 + 2 * i + w;
          const uint4 o = make_uint4(cvt_e4m3x2_f16x2(v[i].x), cvt_e4m3x2_f16x2(v[i].x >> 16),
                                     cvt_e4m3x2_f16x2(v[i].y), cvt_e4m3x2_f16x2(v[i].y >> 16));
          st_shared_v4(dst + bx * kLatBox + r * 128 + ((ch ^ (r & 7)) << 4), o);
        }
      }
      // rope: 8 rows x 4 chunks per warp step
      {
        uint2 v[4];
#pragma unroll
        for (int it = 0; it < 4; ++it) {
          const int r = 16 * it + 8 * w + (lane >> 2), cr = lane & 3;
          v[it] = r < live ? ld_shared_v2(src + kF8RopeOff + r * 32 + cr * 8) : make_uint2(0, 0);
        }
#pragma unroll
        for (int it = 0; it < 4; ++it) {
          const int r = 16 * it + 8 * w + (lane >> 2), cr = lane & 3;
          const uint4 o = make_uint4(cvt_e4m3x2_f16x2(v[it].x), cvt_e4m3x2_f16x2(v[it].x >> 16),
                                     cvt_e4m3x2_f16x2(v[it].y), cvt_e4m3x2_f16x2(v[it].y >> 16));
          st_shared_v4(dst + 4 * kLatBox + r * 64 + ((cr ^ ((r >> 1) & 3)) << 4), o);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(c.bar(B_KV_FULL + os));
      mbar_arrive(c.bar(B_F8_EMPTY + fs));
    }
  }
}



// ------------------------------------------------------------------ MMA issuer

template <class S, bool F8>
__device__ void mma_issuer(const Ctx& c, const S& sched, const DecodeArgs& a, uint32_t tmem, int worker, int role) {
  constexpr int NS = op_stages<F8>();
  constexpr uint32_t kIdescS = idesc_s<F8>(), kIdescPV = idesc_pv<F8>();
  // Two cursors walk this worker's tile sequence: S products run ahead as
  // soon as a cache tile has landed and the S buffer they write was read by
  // the softmax warps; P.V products follow as P tiles appear.  role 0 issues
  // both from this thread (whichever is ready), role 1 only the S products
  // and role 2 only the P.V products, from two threads of different warps:
  // issuing the 18 MMAs of an S product takes a single thread about 0.6 us,
  // and a P tile that became ready meanwhile would wait for it.  The two
  // streams touch disjoint TMEM (S buffers; O) and only read the cache stage;
  // a stage is released after its P.V, which follows its S product (the
  // softmax read that S before forming P).
  const int seg_end = sched.end(worker);
  auto first_live = [&](int s) {
    while (s < seg_end && segment_tiles(sched.seg(s), seg_len(c, sched, a, s)) == 0) ++s;
    return s;
  };
  int s_seg = first_live(sched.begin(worker)), s_jj = 0, s_j = 0, q_used = 0;
  int p_seg = s_seg, p_jj = 0, p_j = 0;
  int s_nt = s_seg < seg_end ? segment_tiles(sched.seg(s_seg), seg_len(c, sched, a, s_seg)) : 0;
  int p_nt = s_nt;
  long long t_last = clock64();
  while (role == 1 ? s_seg < seg_end : p_seg < seg_end) {
    bool progressed = false;
    if (role != 2 && s_seg < seg_end) {
      const int stage = s_j % NS;
      bool ready = (s_jj > 0 || mbar_test_wait(c.bar(B_Q_READY), q_used & 1)) &&
                   mbar_test_wait(c.bar(B_KV_FULL + stage), (s_j / NS) & 1) &&
                   (s_j < 2 || mbar_test_wait(c.bar(B_S_FREE + (s_j & 1)), ((s_j >> 1) - 1) & 1));
      if (ready) {
        if (s_jj == 0) ++q_used;
        tc_fence_after();
        const uint32_t stage_addr = c.sbase + OFF_KV + stage * kStageBytes;
        const uint32_t d = tmem + TM_S + 64 * (s_j & 1);
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
          // B = cache latent half (64 tokens x 256), K-major 128B swizzle
          const uint64_t bdesc = smem_desc(stage_addr + (kk >> 2) * kLatBox + (kk & 3) * 32, 16, 1024, kSwizzle128B);
          mma_ts(d, tmem + TM_Q + 8 * kk, bdesc, kIdescS, kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const uint64_t adesc = smem_desc(c.sbase + OFF_QROPE + kk * 32, 16, 512, kSwizzle64B);
          const uint64_t bdesc = smem_desc(stage_addr + 4 * kLatBox + kk * 32, 16, 512, kSwizzle64B);
          mma_ss(d, adesc, bdesc, kIdescS, 1u);
        }
        mma_commit(c.bar(B_S_FULL + (s_j & 1)));
        ++s_j;
        if (++s_jj == s_nt) {
          s_jj = 0;
          s_seg = first_live(s_seg + 1);
          s_nt = s_seg < seg_end ? segment_tiles(sched.seg(s_seg), seg_len(c, sched, a, s_seg)) : 0;
        }
        progressed = true;
      }
    }
    if (role != 1 && (role == 2 || p_j < s_j) && mbar_test_wait(c.bar(B_P_FULL), p_j & 1)) {
      tc_fence_after();
      const uint32_t stage_addr = c.sbase + OFF_KV + (p_j % NS) * kStageBytes;
      const uint32_t p_addr = c.sbase + OFF_P;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        // A = P (128 rows x 64 keys) K-major 128B swizzle; B = V (keys x 256
        // latent) MN-major 128B swizzle: 64-column atoms 8 KB apart (LBO),
        // 8-key row groups 1 KB apart (SBO)
        const uint64_t adesc = smem_desc(p_addr + kk * 32, 16, 1024, kSwizzle128B);
        const uint64_t bdesc = smem_desc(stage_addr + kk * 16 * 128, kLatBox, 1024, kSwizzle128B);
        mma_ss(tmem + TM_O, adesc, bdesc, kIdescPV, (p_jj == 0 && kk == 0) ? 0u : 1u);
      }
      mma_commit(c.bar(B_PV_DONE));
      mma_commit(c.bar(B_KV_EMPTY + (p_j % NS)));
      ++p_j;
      if (++p_jj == p_nt) {
        p_jj = 0;
        p_seg = first_live(p_seg + 1);
        p_nt = p_seg < seg_end ? segment_tiles(sched.seg(p_seg), seg_len(c, sched, a, p_seg)) : 0;
      }
      progressed = true;
    }
    if (progressed) {
      t_last = clock64();
    } else if (*c.abort_flag) {
      break;
    } else if (clock64() - t_last > kTimeoutCycles) {
      *c.abort_flag = 1;
      atomicCAS(&g_kernel_error, 0, 0x204);
      break;
    }
  }
  // all issued tensor-core work must finish before TMEM is released
  const uint32_t fin = c.bar(role == 2 ? B_FINAL2 : B_FINAL);
  mma_commit(fin);
  const long long t0 = clock64();
  while (!mbar_try_wait(fin, 0) && clock64() - t0 < kTimeoutCycles) {
  }
}

// ------------------------------------------------------------------ softmax

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi, float& rlo, float& rhi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  rlo = __low2float(v);
  rhi = __high2float(v);
  return *reinterpret_cast<uint32_t*>(&v);
}

// ------------------------------------------------------------------ exchange

// Partial scores cross to the peer as 24-bit codes: the float's top 24 bits
// (sign, exponent, 15 mantissa bits).  Rounding is one multiply and a
// truncation: x * (1 + 85 * 2^-23) adds between 0.332 and 0.664 of a code unit
// to |x| (in proportion to the mantissa), so the dropped bits round the kept
// ones with an error of at most 0.668 of a code unit, a relative error below
// (4/3) * 2^-16.  Because it is a floating-point multiply, every NaN becomes
// the canonical NaN (top bits all ones, still a NaN after the truncation) and
// infinities stay infinite, so both CTAs of the pair see the same non-finite
// score; an integer rounding add would carry the canonical NaN's mantissa into
// the sign bit.  Four codes fill three words.
constexpr float kCodeRound = 1.00001013278961181640625f;  // 1 + 85 * 2^-23, exact in float32
__device__ __forceinline__ uint32_t score24(uint32_t bits) {
  return __float_as_uint(__uint_as_float(bits) * kCodeRound) >> 8;
}
__device__ __forceinline__ void pack24(const uint32_t* v, uint32_t* w) {
  const uint32_t a = score24(v[0]), b = score24(v[1]), c = score24(v[2]), d = score24(v[3]);
  w[0] = a | (b << 24);
  w[1] = (b >> 8) | (c << 16);
  w[2] = (c >> 16) | (d << 8);
}
__device__ __forceinline__ void unpack24(const uint32_t* w, float* v) {
  v[0] = __uint_as_float(w[0] << 8);
  v[1] = __uint_as_float(((w[0] >> 24) | (w[1] << 8)) << 8);
  v[2] = __uint_as_float(((w[1] >> 16) | (w[2] << 16)) << 8);
  v[3] = __uint_as_float((w[2] >> 8) << 8);
}

// Warps 12-15 (one per TMEM lane quadrant, thread = query row): as soon as a
// tile's partial scores land in TMEM, copy them to registers and stream them
// into the peer CTA's receive buffer with st.async, which completes bytes on
// the peer's x_full barrier.  Decoupled from the softmax warps so that the
// time it takes to issue 24 KB of remote stores per tile never blocks them.
// bf16 pair -> fp16 pair (exact for values in fp16's normal range, which
// covers any sane query; used for the fp16 operands of the e4m3 path)
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
  __half2 h = __floats2half2_rn(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
  return *reinterpret_cast<uint32_t*>(&h);
}

template <class S, bool F8, bool Q8>
__device__ void exchanger(const Ctx& c, const S& sched, const DecodeArgs& a, uint32_t tmem, int worker,
                          int rank) {
  const int quad = (threadIdx.x >> 5) & 3;
  const int lane = threadIdx.x & 31;
  const int row = quad * 32 + lane;
  const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
  const uint32_t peer = rank ^ 1;
  const uint32_t xchg_peer = mapa(c.sbase + OFF_XCHG, peer) + row * 16;
  const uint32_t x_full_peer = mapa(c.bar(B_X_FULL), peer);  // slot k's barrier at + 8k
  const int M = a.rows;
  const bool valid_row = row < M;  // padding rows (M < 128) exchange nothing
  // A warp whose rows are all padding sends nothing, so it must not wait on
  // the "read" notes either: those phases are paced by the live rows alone
  // and could run two phases ahead of it (a parity wait would then hang).
  const bool warp_live = 32 * quad < M;
  int j = 0;
  bool ok = true;
  for (int s = sched.begin(worker); ok && s < sched.end(worker); ++s) {
    const Segment sg = sched.seg(s);
    const int nt = segment_tiles(sg, seg_len(c, sched, a, s));
    if (nt == 0) continue;
    // ---- this segment's query: latent half -> TMEM columns [384, 512), rope
    // half -> shared memory (64B swizzle).  The previous segment's S MMAs all
    // completed (this warp waited for each), so the old Q and the rope area
    // are dead; the load overlaps the softmax warps' last tile and epilogue.
    // Loads are coalesced: four lanes read one 64-byte piece of a row, eight
    // rows per instruction.  Each 64-byte column piece of the warp's 32 rows
    // is staged through this warp's 2 KB of the rope area (XOR-swizzled by
    // row pair, conflict-free both ways) so that lane r can store row r's
    // piece into TMEM; the rope rows go straight to their final layout.
    {
      const int ql = lane >> 2, qc = lane & 3;  // load mapping: row 8k + ql, 16-byte chunk qc
      const int2 q = seg_q(c, sched, a, s);
      const int rows_b = q.y * a.num_heads;     // this request's query rows (<= M; the rest stay 0)
      const size_t row0 = (size_t)q.x * a.num_heads + 32 * quad;
      const uint4* qn = reinterpret_cast<const uint4*>(a.q_nope) + row0 * (kLatent / 8) + 32 * rank + qc;
      const uint4* qp = reinterpret_cast<const uint4*>(a.q_pe) + row0 * (kRope / 8) + 4 * rank + qc;
      // e4m3 query (Q8): merged [row][576] bytes; this lane's 8 columns are 8 bytes
      const uint2* q8 = reinterpret_cast<const uint2*>(a.q_nope) + row0 * (kKvDim / 8) + 32 * rank + qc;
      const uint32_t stage = c.sbase + OFF_QROPE + quad * 2048;  // this warp's rows of the rope area
      auto lrow_ok = [&](int rl) { return 32 * quad + rl < rows_b; };
      // 8 e4m3 values -> 8 fp16 (exact)
      auto widen = [&](uint2 v) {
        return make_uint4(cvt_e4m3x2_f16x2(v.x), cvt_e4m3x2_f16x2(v.x >> 16), cvt_e4m3x2_f16x2(v.y),
                          cvt_e4m3x2_f16x2(v.y >> 16));
      };
      // 8 latent columns of row rl, chunk cidx (8-column units within this CTA's half)
      auto load_lat = [&](int rl, int cidx) {
        if (!lrow_ok(rl)) return make_uint4(0, 0, 0, 0);
        if (Q8) return widen(__ldg(q8 + (size_t)rl * (kKvDim / 8) + cidx));
        return __ldg(qn + (size_t)rl * (kLatent / 8) + cidx);
      };
      auto load_rope = [&](int rl) {
        if (!lrow_ok(rl)) return make_uint4(0, 0, 0, 0);
        if (Q8) return widen(__ldg(q8 + (size_t)rl * (kKvDim / 8) + (kLatent / 8) - 28 * rank));
        return __ldg(qp + (size_t)rl * (kRope / 8));
      };
      // bf16 -> fp16 for the e4m3 cache's fp16 MMAs (an e4m3 query is fp16 already)
      auto cvt4 = [&](uint4 v) {
        return (F8 && !Q8)
                   ? make_uint4(bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y), bf16x2_to_f16x2(v.z), bf16x2_to_f16x2(v.w))
                   : v;
      };
      uint4 rpe[4], lat[4][4];
#pragma unroll
      for (int rd = 0; rd < 4; ++rd)
#pragma unroll
        for (int k = 0; k < 4; ++k) lat[rd][k] = load_lat(8 * k + ql, 4 * rd);
      // piece p (0..7) = latent columns [32p, 32p+32) of this CTA's half =
      // TMEM columns TM_Q + 16p; piece p + 4 is requested as piece p retires
#pragma unroll
      for (int pc = 0; pc < 8; ++pc) {
        const int rd = pc & 3;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int rl = 8 * k + ql;
          st_shared_v4(stage + rl * 64 + ((qc ^ ((rl >> 1) & 3)) << 4), lat[rd][k]);
        }
        __syncwarp();
        if (pc < 4) {
#pragma unroll
          for (int k = 0; k < 4; ++k) lat[rd][k] = load_lat(8 * k + ql, 4 * (rd + 4));
        } else if (pc == 4) {
#pragma unroll
          for (int k = 0; k < 4; ++k) rpe[k] = load_rope(8 * k + ql);
        }
        uint32_t r[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 v = cvt4(ld_shared_v4(stage + lane * 64 + ((i ^ ((lane >> 1) & 3)) << 4)));
          r[4 * i + 0] = v.x; r[4 * i + 1] = v.y; r[4 * i + 2] = v.z; r[4 * i + 3] = v.w;
        }
        tmem_st16(tmem + lane_off + TM_Q + 16 * pc, r);
        __syncwarp();
      }
      // rope rows of this warp in the MMA's 64B-swizzled layout (row-pair
      // XOR of the 16-byte chunk: the same pattern as the staging)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int rl = 8 * k + ql;
        st_shared_v4(stage + rl * 64 + ((qc ^ ((rl >> 1) & 3)) << 4), cvt4(rpe[k]));
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(c.bar(B_Q_READY));
    }
    for (int jj = 0; jj < nt; ++jj, ++j) {
      const int sb = j & 1, u = j >> 1;
      if (!wait_bar_warp<false>(c, c.bar(B_S_FULL + sb), u & 1, 0x401)) { ok = false; break; }
      tc_fence_after();
      uint32_t sv64[64];
      tmem_ld64(tmem + lane_off + TM_S + 64 * sb, sv64);
      tc_fence_before();
      mbar_arrive(c.bar(B_S_LOADED + sb));
      // the two 32-key halves go to ring slots (2j) % 3 and (2j + 1) % 3;
      // a slot's previous half must have been read by the peer
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int g = 2 * j + h, k = g % kSlots, ug = g / kSlots;
        if (warp_live && ug > 0 && !wait_bar_warp<true>(c, c.bar(B_X_EMPTY + k), (ug - 1) & 1, 0x402)) {
          ok = false;
          break;
        }
        const uint32_t dst = xchg_peer + k * kSlotBytes;
        const uint32_t mb = x_full_peer + 8 * k;
        const uint32_t* sv = sv64 + 32 * h;
        if (valid_row) {
          uint32_t w[24];
#pragma unroll
          for (int q = 0; q < 8; ++q) pack24(sv + 4 * q, w + 3 * q);
#pragma unroll
          for (int ch = 0; ch < kXchgChunks; ++ch)
            st_async_v4(dst + ch * 2048, w[4 * ch], w[4 * ch + 1], w[4 * ch + 2], w[4 * ch + 3], mb);
        }
        // arm the "peer has read it" phase of this slot: one 4-byte note per live row
        if (threadIdx.x == 384) mbar_arrive_expect_tx(c.bar(B_X_EMPTY + k), 4 * M);
      }
      if (!ok) break;
    }
  }
  // drain: the peer's notes for the last half tiles are the only remote
  // writes nothing else waits for; they must land before this CTA may exit
  // (half tile g sits in slot g % kSlots, phase g / kSlots)
  for (int g = 2 * j - 1; warp_live && ok && g >= 0 && g >= 2 * j - kSlots; --g)
    if (!wait_bar_warp<true>(c, c.bar(B_X_EMPTY + g % kSlots), (g / kSlots) & 1, 0x403)) break;
}

template <class S, bool F8>
__device__ void softmax_epilogue(const Ctx& c, const S& sched, const DecodeArgs& a, uint32_t tmem,
                                 int worker, int rank) {
  // Two warps per TMEM lane quadrant: warp (4 + q) and (8 + q) own query rows
  // 32q..32q+31 (= TMEM lanes); `half` selects which 32 of a tile's 64 keys
  // (and which 128 of this CTA's 256 output columns) the thread handles.
  const int sw = (threadIdx.x >> 5) - 4;
  const int quad = (threadIdx.x >> 5) & 3;
  const int half = sw >> 2;
  const int row = quad * 32 + (threadIdx.x & 31);
  const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
  const uint32_t peer = rank ^ 1;
  const int M = a.rows;
  const bool valid_row = row < M;
  // A warp whose rows are all padding reads nothing from the exchange and
  // sends no "read" note: it must not wait on the receive barriers, whose
  // phases are paced by the live rows' notes alone and could run two phases
  // ahead of it (its parity wait would then hang).  Its rows see no key.
  const bool warp_live = 32 * quad < M;
  const int qi = valid_row ? row / a.num_heads : 0;  // query position of this row
  // Exchange ring slots hold [16-byte chunk][row] so a warp's stores are
  // contiguous; half tile g = 2j + half of this thread sits in slot g % 3.
  const uint32_t xchg_local = c.sbase + OFF_XCHG + row * 16;
  const uint32_t x_empty_peer = mapa(c.bar(B_X_EMPTY), peer);  // slot k's barrier at + 8k
  const uint32_t sink_peer = mapa(c.sbase + OFF_SINK, peer) + row * 4;
  const uint32_t rearm_thread = 128 + 128 * half;  // re-arms this half's slots
  float* red_max = reinterpret_cast<float*>(c.smem + OFF_RED);      // [2 tiles][2 halves][128]
  float* red_l = red_max + 2 * 2 * 128;                              // [2 segments][2 halves][128]
  const float cs = a.score_scale_log2;  // raw score -> base-2 logit
  int j = 0, nseg = 0;
  bool ok = true;
  // leaving early: release the quadrant's other warp from the named barrier
  // it may be waiting at, now or one tile later
  auto bail = [&]() {
    named_bar_arrive(1 + quad, 64);
    named_bar_arrive(1 + quad, 64);
  };

  for (int s = sched.begin(worker); ok && s < sched.end(worker); ++s) {
    const Segment sg = sched.seg(s);
    const int L = seg_len(c, sched, a, s);
    const int nt = segment_tiles(sg, L);
    // visible keys of this row; rows past the request's query rows (ragged
    // batches) still take part in the exchange with the peer but see no key
    // and write nothing
    int vis;
    {
      const int2 q = seg_q(c, sched, a, s);
      vis = row < q.y * a.num_heads ? L - q.y + 1 + qi : 0;
    }
    float m_ref = -CUDART_INF_F, l = 0.f;

    if (nt > 0) {

      for (int jj = 0; jj < nt; ++jj, ++j) {
        const int sb = j & 1;
        // ---- own partial scores: the exchange warps have read S out of
        // TMEM (so P may overwrite it later); this thread's 32 columns
        if (!wait_bar_warp<false>(c, c.bar(B_S_LOADED + sb), (j >> 1) & 1, 0x301)) { ok = false; bail(); break; }
        tc_fence_after();
        uint32_t cur[32];
        // issued now, completed after the peer's half is read: the two latencies overlap
        tmem_ld32_async(tmem + lane_off + TM_S + 64 * sb + 32 * half, cur);
        // ---- full scores: own partial + the peer's (its st.async bytes
        // complete the transaction count armed for this phase).  Re-arming
        // the next phase right away is safe: the peer cannot send into this
        // slot again before all "read" notes of this phase reached it.
        const int g = 2 * j + half, slot = g % kSlots, ug = g / kSlots;
        if (warp_live && !wait_bar_warp<true>(c, c.bar(B_X_FULL + slot), ug & 1, 0x303)) {
          tmem_wait_ld32(cur);
          ok = false;
          bail();
          break;
        }
        if (threadIdx.x == rearm_thread) mbar_arrive_expect_tx(c.bar(B_X_FULL + slot), kXchgRowBytes * M);  // row 0: live
        float x[32];
        if (!warp_live) {
          tmem_wait_ld32(cur);
          tc_fence_before();
          mbar_arrive(c.bar(B_S_FREE + sb));  // the MMA may overwrite this S buffer
#pragma unroll
          for (int k = 0; k < 32; ++k) x[k] = __uint_as_float(cur[k]);  // masked below: no visible key
        } else {
          const uint32_t srcx = xchg_local + slot * kSlotBytes;
          uint32_t w[24];
#pragma unroll
          for (int ch = 0; ch < kXchgChunks; ++ch) {
            const uint4 v = ld_shared_v4(srcx + ch * 2048);
            w[4 * ch + 0] = v.x; w[4 * ch + 1] = v.y; w[4 * ch + 2] = v.z; w[4 * ch + 3] = v.w;
          }
          tmem_wait_ld32(cur);
          tc_fence_before();
          mbar_arrive(c.bar(B_S_FREE + sb));  // the MMA may overwrite this S buffer
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            float pv[4];
            unpack24(w + 3 * q, pv);
#pragma unroll
            for (int t = 0; t < 4; ++t) x[4 * q + t] = __uint_as_float(cur[4 * q + t]) + pv[t];
          }
        }
        // ---- causal / length mask (tail tiles only), row max over both
        // halves on the raw scores (the scale is positive)
        const int nvis = vis - ((sg.tile_begin + jj) * kTileTokens + 32 * half);
        if (nvis < 32) {
#pragma unroll
          for (int k = 0; k < 32; ++k) x[k] = k < nvis ? x[k] : -CUDART_INF_F;
        }
        float mt;
        {
          float m16[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) m16[k] = fmaxf(x[k], x[k + 16]);
#pragma unroll
          for (int k = 0; k < 8; ++k) m16[k] = fmaxf(m16[k], m16[k + 8]);
#pragma unroll
          for (int k = 0; k < 4; ++k) m16[k] = fmaxf(m16[k], m16[k + 4]);
          mt = fmaxf(fmaxf(m16[0], m16[2]), fmaxf(m16[1], m16[3]));
        }
        // tell the peer its buffer is free: a 4-byte st.async whose value (the
        // row max) depends on every word read from the buffer
        if (valid_row) st_async_b32(sink_peer + slot * kNoteBytes, __float_as_uint(mt), x_empty_peer + 8 * slot);
        red_max[(sb * 2 + half) * 128 + row] = mt;
        named_bar_sync(1 + quad, 64);  // the quadrant's two warps swap row maxima (hardware barrier 1 + quad)
        mt = fmaxf(red_max[(sb * 2) * 128 + row], red_max[(sb * 2 + 1) * 128 + row]) * cs;
        // lazy rescale: the reference max moves only when it grew by more than
        // 2^8; both halves decide identically.  The decision and P need only
        // S, so they are formed while the previous tile's P.V still runs.
        const float m_new = fmaxf(m_ref, mt);
        const bool resc = m_new > m_ref + kRescaleThreshold;
        const float alpha = resc ? ex2_approx(m_ref - m_new) : 1.f;  // 0 when m_ref = -inf
        if (resc) {
          l *= alpha;
          m_ref = m_new;
        }
        const float nm = m_ref == -CUDART_INF_F ? 0.f : -m_ref;  // all-masked rows: 2^-inf = 0
        // ---- P as bf16 (fp16 for a float8 cache) pairs in registers
        uint32_t pk[16];
        float lsum = 0.f;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float p0 = ex2_approx(fmaf(x[2 * k], cs, nm));
          const float p1 = ex2_approx(fmaf(x[2 * k + 1], cs, nm));
          if (F8) {
            __half2 hv = __floats2half2_rn(p0, p1);
            pk[k] = *reinterpret_cast<uint32_t*>(&hv);
          } else {
            float r0, r1;
            pk[k] = pack_bf16(p0, p1, r0, r1);
          }
          lsum += p0 + p1;  // l from the unrounded probabilities: exact lse
        }
        l += lsum;
        // ---- O and the P buffer are idle once the previous tile's P.V is
        // done; a rescale of O is TMEM traffic by whole warps
        if (jj > 0) {
          if (!wait_bar_warp<false>(c, c.bar(B_PV_DONE), (j - 1) & 1, 0x304)) { ok = false; bail(); break; }
          tc_fence_after();
          if (__any_sync(0xffffffffu, resc)) {
#pragma unroll 1
            for (int ck = 0; ck < 4; ++ck) {
              uint32_t o[32];
              const uint32_t addr = tmem + lane_off + TM_O + 128 * half + 32 * ck;
              tmem_ld32(addr, o);
#pragma unroll
              for (int v = 0; v < 32; ++v) o[v] = __float_as_uint(__uint_as_float(o[v]) * alpha);
              tmem_st32(addr, o);
            }
          }
        }
        // ---- P to shared memory, K-major 128B swizzle: this thread's 32 keys
        // are 16-byte chunks 4*half..4*half+3 of its row
        {
          const uint32_t prow = c.sbase + OFF_P + row * 128;
#pragma unroll
          for (int i = 0; i < 4; ++i)
            st_shared_v4(prow + (((4 * half + i) ^ (row & 7)) << 4),
                         make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]));
        }
        fence_proxy_async_smem();
        tc_fence_before();  // orders a rescale's TMEM stores to O before the P.V that follows
        mbar_arrive(c.bar(B_P_FULL));
      }
      if (!ok) break;
      if (!wait_bar_warp<false>(c, c.bar(B_PV_DONE), (j - 1) & 1, 0x305)) { ok = false; bail(); break; }
      tc_fence_after();
    }

    // ---- epilogue: row sum over both halves; this thread writes 128 of the
    // CTA's 256 output columns, (rank 0, half 0) the lse.  TMEM is read by
    // whole warps (only when the segment ran MMAs); stores are per row.
    {
      float* rl = red_l + (nseg & 1) * 256;
      rl[half * 128 + row] = l;
      mbar_arrive(c.bar(B_PAIR_L + quad));
      if (!wait_bar_warp<false>(c, c.bar(B_PAIR_L + quad), nseg & 1, 0x307)) { ok = false; bail(); break; }
      l = rl[row] + rl[128 + row];
      ++nseg;
    }
    {
      // output row of this thread's query row, -1 past the request's rows
      // (re-read from the cache: nothing is held across the tile loop)
      const int orow = out_row(seg_q(c, sched, a, s), a.num_heads, row);
      const bool live_row = orow >= 0;
      // l = 0 only for a row that saw no key; a NaN score (NaN in a visible
      // cache row or in the query) leaves l NaN and the row NaN, as in the
      // definition
      const bool live = !(l == 0.f);
      const float inv = live ? a.out_scale / l : 0.f;
#pragma unroll 1
      for (int ck = 0; ck < 4; ++ck) {
        uint32_t o[32];
        if (nt > 0) {
          tmem_ld32(tmem + lane_off + TM_O + 128 * half + 32 * ck, o);
        }
        if (nt == 0 || !live) {
#pragma unroll
          for (int v = 0; v < 32; ++v) o[v] = 0u;
        }
        const int col = 256 * rank + 128 * half + 32 * ck;
        if (sg.slot < 0 ? !live_row : !valid_row) continue;
        if (sg.slot < 0) {
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) + (size_t)orow * kLatent + col);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            float d0, d1;
            uint4 w;
            w.x = pack_bf16(__uint_as_float(o[8 * v + 0]) * inv, __uint_as_float(o[8 * v + 1]) * inv, d0, d1);
            w.y = pack_bf16(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv, d0, d1);
            w.z = pack_bf16(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv, d0, d1);
            w.w = pack_bf16(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv, d0, d1);
            dst[v] = w;
          }
        } else {
          // partials are bf16, chunk-major [slot][8-column chunk][row]: a
          // warp's 32 rows store 512 contiguous bytes per chunk
          uint4* dst = reinterpret_cast<uint4*>(a.part_o) + ((size_t)sg.slot * (kLatent / 8) + col / 8) * M + row;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            float d0, d1;
            uint4 w;
            w.x = pack_bf16(__uint_as_float(o[8 * v + 0]) * inv, __uint_as_float(o[8 * v + 1]) * inv, d0, d1);
            w.y = pack_bf16(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv, d0, d1);
            w.z = pack_bf16(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv, d0, d1);
            w.w = pack_bf16(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv, d0, d1);
            dst[(size_t)v * M] = w;
          }
        }
      }
      if (rank == 0 && half == 0 && valid_row) {
        const float lse = live ? (m_ref + __log2f(l)) * 0.6931471805599453f : -CUDART_INF_F;
        if (sg.slot < 0) {
          if (live_row) a.lse[orow] = lse;
        } else {
          a.part_lse[(size_t)sg.slot * M + row] = lse;
        }
      }
    }
    tc_fence_before();
  }
}

// ------------------------------------------------------------------ kernel

template <class R, bool F8, bool Q8>
__device__ __forceinline__ void run_roles(const Ctx& c, const R& sched, const DecodeArgs& a, uint32_t tmem,
                                          int worker, int rank, int warp, const CUtensorMap& tm_lat,
                                          const CUtensorMap& tm_rope) {
  if (warp == 0) {
    producer<R, F8, Q8>(c, sched, a, &tm_lat, &tm_rope, worker, rank);
  } else if (warp == 1) {
    if ((threadIdx.x & 31) == 0) mma_issuer<R, F8>(c, sched, a, tmem, worker, F8 ? 0 : 1);
    __syncwarp();
  } else if (!F8 && warp == 3) {
    if ((threadIdx.x & 31) == 0) mma_issuer<R, F8>(c, sched, a, tmem, worker, 2);
    __syncwarp();
  } else if (warp >= 12) {
    exchanger<R, F8, Q8>(c, sched, a, tmem, worker, rank);
  } else if (warp >= 4) {
    softmax_epilogue<R, F8>(c, sched, a, tmem, worker, rank);
  } else if (F8) {
    converter<R>(c, sched, a, worker);
  }
}

// The whole kernel; `sched` is a kernel parameter (host plan) or lives in the
// workspace (device plan, kDevSched: written by the planner grid that runs
// just before, so it is read only after griddepcontrol.wait).
template <class S, bool F8, bool kDevSched, bool Q8>
__device__ __forceinline__ void decode_body(const S& sched, const DecodeArgs& a,
                                            const CUtensorMap& tm_lat, const CUtensorMap& tm_rope) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  Ctx c;
  c.smem = smem_raw + pad;
  c.sbase = raw + pad;
  c.abort_flag = reinterpret_cast<volatile int*>(c.smem + OFF_ABORT);
  const int warp = threadIdx.x >> 5;
  const int rank = (int)cluster_ctarank();
  const int worker = blockIdx.x >> 1;
  c.seg_len = reinterpret_cast<const int*>(c.smem + OFF_SEGLEN);
  c.seg_q = reinterpret_cast<const int2*>(c.smem + OFF_SEGQ);
  // key counts and query rows of this worker's segments (and, for a device
  // plan, the segments themselves), read once for every role
  auto read_schedule = [&]() {
    c.seg0 = worker < sched.num_workers() ? sched.begin(worker) : 0;
    if (warp == 2 && worker < sched.num_workers()) {
      const int n = min(sched.end(worker) - c.seg0, kSegLenCache);
      for (int i = threadIdx.x & 31; i < n; i += 32) {
        const Segment sg = sched.seg(c.seg0 + i);
        reinterpret_cast<int*>(c.smem + OFF_SEGLEN)[i] = request_len(a, sg.req);
        reinterpret_cast<int2*>(c.smem + OFF_SEGQ)[i] = request_q_checked(a, sg.req);
        if (kDevSched) reinterpret_cast<Segment*>(c.smem + OFF_SEGS)[i] = sg;
      }
    }
  };
  if (!kDevSched) read_schedule();

  if (threadIdx.x == 0) {
    *c.abort_flag = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(c.bar(B_KV_FULL + s), F8 ? 64 : 1);  // e4m3: the 64 converter threads
      mbar_init(c.bar(B_KV_EMPTY + s), 1);
      mbar_init(c.bar(B_F8_FULL + s), 1);
      mbar_init(c.bar(B_F8_EMPTY + s), 64);
    }
    for (int i = 0; i < 2; ++i) mbar_init(c.bar(B_S_FULL + i), 1);
    mbar_init(c.bar(B_P_FULL), 256);
    for (int k = 0; k < kSlots; ++k) {
      mbar_init(c.bar(B_X_FULL + k), 1);   // own expect_tx arrival + the peer's st.async bytes
      mbar_init(c.bar(B_X_EMPTY + k), 1);  // own expect_tx arrival + the peer's 4-byte notes
    }
    mbar_init(c.bar(B_PV_DONE), 1);
    mbar_init(c.bar(B_Q_READY), 128);
    mbar_init(c.bar(B_TAIL), 1);
    mbar_init(c.bar(B_FINAL), 1);
    mbar_init(c.bar(B_FINAL2), 1);
    // receive buffers are armed one phase ahead: phase 0 now, phase u+1 as
    // soon as phase u completed (so the peer's bytes never precede the arm)
    for (int k = 0; k < kSlots; ++k) mbar_arrive_expect_tx(c.bar(B_X_FULL + k), kXchgRowBytes * a.rows);
    for (int i = 0; i < 4; ++i) mbar_init(c.bar(B_PAIR_L + i), 64);
    for (int i = 0; i < 2; ++i) mbar_init(c.bar(B_S_LOADED + i), 128);
    for (int i = 0; i < 2; ++i) mbar_init(c.bar(B_S_FREE + i), 256);
    fence_mbar_init();
    prefetch_tensormap(&tm_lat);
    prefetch_tensormap(&tm_rope);
  }
  if (warp == 1) {
    tmem_alloc(c.sbase + OFF_TMEM_SLOT, kTmemCols);
    tmem_relinquish();
  }
  // device plan: all of the above overlapped the planner grid; the schedule
  // is complete and visible once this returns
  if (kDevSched) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    read_schedule();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // peer barriers initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(c.smem + OFF_TMEM_SLOT);

  if (worker < sched.num_workers()) {
    if (kDevSched) {
      const int last = sched.end(worker);
      const CachedSched cs{static_cast<const Schedule<kSegCapLarge>*>(sched.raw()),
                           reinterpret_cast<const Segment*>(c.smem + OFF_SEGS), c.seg0, last,
                           min(last - c.seg0, kSegLenCache), sched.num_workers()};
      run_roles<CachedSched, F8, Q8>(c, cs, a, tmem, worker, rank, warp, tm_lat, tm_rope);
    } else {
      run_roles<S, F8, Q8>(c, sched, a, tmem, worker, rank, warp, tm_lat, tm_rope);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // every global write of this CTA is issued: a programmatic dependent
  // (the combine) may be scheduled once all CTAs got here; it still waits
  // for this grid's completion before it reads anything
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
  cluster_sync();  // no peer may still write into this CTA's shared memory
}

template <int CAP, bool F8, bool Q8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ Schedule<CAP> sched, const __grid_constant__ DecodeArgs a,
                  const __grid_constant__ CUtensorMap tm_lat, const __grid_constant__ CUtensorMap tm_rope) {
  decode_body<ParamSched<CAP>, F8, false, Q8>(ParamSched<CAP>{sched}, a, tm_lat, tm_rope);
}

// Device-planned variant: the schedule is in the workspace.
template <bool F8, bool Q8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_kernel_dev(const Schedule<kSegCapLarge>* sched, const __grid_constant__ DecodeArgs a,
                      const __grid_constant__ CUtensorMap tm_lat, const __grid_constant__ CUtensorMap tm_rope) {
  decode_body<GlobalSched, F8, true, Q8>(GlobalSched{sched}, a, tm_lat, tm_rope);
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D view [num_pages * page_size rows, 576 columns] of the cache (bf16 or
// one-byte e4m3 elements).
static bool make_map(CUtensorMap* m, const void* kv, int64_t rows, int box_cols, int box_rows,
                     CUtensorMapSwizzle sw, bool fp8) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kKvDim, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kKvDim * (fp8 ? 1 : 2)};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                  const_cast<void*>(kv), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int CAP, bool F8, bool Q8>
static cudaError_t launch_cap(const mla_plan& p, const DecodeArgs& a, const CUtensorMap& lat,
                              const CUtensorMap& rope, cudaStream_t stream) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err =
        cudaFuncSetAttribute(decode_kernel<CAP, F8, Q8>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  });
  if (attr_err != cudaSuccess) return attr_err;
  Schedule<CAP> s;
  s.num_workers = p.num_workers;
  s.num_segments = (int32_t)p.segs.size();
  for (int w = 0; w <= p.num_workers; ++w) s.worker_seg[w] = p.worker_seg[w];
  for (size_t i = 0; i < p.segs.size(); ++i) s.seg[i] = p.segs[i];
  decode_kernel<CAP, F8, Q8><<<dim3(2 * p.num_workers), kThreads, kSmemBytes, stream>>>(s, a, lat, rope);
  return cudaGetLastError();
}

// Device plan: the schedule sits at the head of the workspace, written by the
// planner grid launched just before on the same stream; this launch is its
// programmatic dependent (see decode_body).
template <bool F8, bool Q8>
static cudaError_t launch_dev(const mla_plan& p, const DecodeArgs& a, const CUtensorMap& lat,
                              const CUtensorMap& rope, const void* workspace, cudaStream_t stream) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(decode_kernel_dev<F8, Q8>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const auto* sched = reinterpret_cast<const Schedule<kSegCapLarge>*>(static_cast<const char*>(workspace) +
                                                                       kDevSchedOffset);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * p.num_workers);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_kernel_dev<F8, Q8>, sched, a, lat, rope);
}

template <bool F8, bool Q8>
static cudaError_t launch_dtype(const mla_plan& p, const DecodeArgs& a, const void* workspace,
                                cudaStream_t stream) {
  CUtensorMap lat, rope;
  const int64_t rows = a.num_pages * a.page_size;
  // bf16: four 64-column 128B-swizzled latent boxes + one 32-column 64B-swizzled
  // rope box per page piece; e4m3: one raw 256-byte latent box + one 32-byte
  // rope box, unswizzled (the converter warps lay out the operands)
  const bool ok = F8 ? make_map(&lat, a.kv, rows, 256, a.page_size, CU_TENSOR_MAP_SWIZZLE_NONE, true) &&
                           make_map(&rope, a.kv, rows, 32, a.page_size, CU_TENSOR_MAP_SWIZZLE_NONE, true)
                     : make_map(&lat, a.kv, rows, 64, a.page_size, CU_TENSOR_MAP_SWIZZLE_128B, false) &&
                           make_map(&rope, a.kv, rows, 32, a.page_size, CU_TENSOR_MAP_SWIZZLE_64B, false);
  if (!ok) return cudaErrorNotSupported;
  if (p.device) return launch_dev<F8, Q8>(p, a, lat, rope, workspace, stream);
  if (p.segs.size() <= (size_t)kSegCapSmall) return launch_cap<kSegCapSmall, F8, Q8>(p, a, lat, rope, stream);
  return launch_cap<kSegCapLarge, F8, Q8>(p, a, lat, rope, stream);
}

}  // namespace sm103

// Returns cudaErrorNotSupported when the tensor-map encoder is unavailable.
// `workspace` is read only for a device plan (its schedule area).
cudaError_t launch_sm103(const mla_plan& p, const DecodeArgs& a, const void* workspace, cudaStream_t stream) {
  // the e4m3 query exists only with an e4m3 cache (the pages' FP8 path)
  if (a.q_e4m3) return sm103::launch_dtype<true, true>(p, a, workspace, stream);
  return a.kv_dtype == MLA_KV_E4M3 ? sm103::launch_dtype<true, false>(p, a, workspace, stream)
                                   : sm103::launch_dtype<false, false>(p, a, workspace, stream);
}

// Kernel-side error code recorded since the last reset (0 = none).
cudaError_t sm103_read_error(int* code, bool reset) {
  cudaError_t e = cudaMemcpyFromSymbol(code, sm103::g_kernel_error, sizeof(int));
  if (e != cudaSuccess || !reset) return e;
  const int zero = 0;
  return cudaMemcpyToSymbol(sm103::g_kernel_error, &zero, sizeof(int));
}

}  // namespace mla
