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
//                                           distributed shared memory)
//   P   = exp2(S * scale*log2e - m)         (both CTAs compute the same P)
//   O_r += P . c_kv[:, half r]              (M = 128, N = 256, K = 64) -> TMEM
// The cache tile in shared memory serves both products: K-major as the B
// operand of S, MN-major as the B operand of P.V.  The 128 query rows
// (heads x q_len, zero-padded) are the M dimension of every MMA.
//
// TMEM (512 columns): O [0,256), S double buffer [256,320) / [320,384) (P is
// written over the S it came from, as bf16 pairs), Q latent half [384,512).
// Shared memory: 4-stage cache-tile ring (36 KB per stage), the rope half of
// Q (8 KB), two 32 KB score-exchange buffers written by the peer CTA.
//
// Warp roles (384 threads): warp 0 TMA producer, warp 1 TMEM allocator and
// MMA issuer, warps 4-11 softmax / correction / epilogue (two warps per query
// row block = TMEM lane quadrant, each owning half of a tile's keys and half
// of the output columns), warps 2-3 spare.  Every wait is bounded: on timeout the kernel
// records an error code in device memory, stops every role, waits for its
// own copies and MMAs, frees TMEM and returns.
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

constexpr int kThreads = 384;  // warps 0-3: producer, MMA, 2 spare; 4-11: softmax
constexpr int kStages = 4;
constexpr int kLatBox = 64 * 128;           // 64 tokens x 64 bf16 columns, 128B swizzle
constexpr int kRopeBox = 64 * 64;           // 64 tokens x 32 bf16 columns, 64B swizzle
constexpr int kStageBytes = 4 * kLatBox + kRopeBox;  // 36864
constexpr int kStageTx = kStageBytes;       // bytes TMA delivers per tile
constexpr int OFF_KV = 0;
constexpr int OFF_QROPE = kStages * kStageBytes;       // 128 rows x 64 B
constexpr int OFF_XCHG = OFF_QROPE + 128 * 64;         // 2 x (128 rows x 256 B)
constexpr int kXchgBytes = 128 * 64 * 4;
constexpr int OFF_RED = OFF_XCHG + 2 * kXchgBytes;     // row max / row sum exchange, 4 KB
constexpr int OFF_SINK = OFF_RED + 4 * 2 * 128 * 4;    // 2 x 256 words the peer's "read done" notes land in
constexpr int kNoteBytes = 256 * 4;
constexpr int OFF_BAR = OFF_SINK + 2 * kNoteBytes;
enum Bar : int {
  B_KV_FULL = 0, B_KV_EMPTY = B_KV_FULL + kStages, B_S_FULL = B_KV_EMPTY + kStages, B_P_FULL = B_S_FULL + 2,
  B_PV_DONE = B_P_FULL + 2, B_Q_READY, B_X_FULL, B_X_EMPTY = B_X_FULL + 2, B_TAIL = B_X_EMPTY + 2, B_FINAL,
  B_PAIR_MAX,                 // [quad][tile parity]: the two warps of a quadrant swap row maxima
  B_PAIR_L = B_PAIR_MAX + 8,  // [quad]: ... and row sums at a segment's end
  B_COUNT = B_PAIR_L + 4
};
constexpr int OFF_TMEM_SLOT = OFF_BAR + B_COUNT * 8;
constexpr int OFF_ABORT = OFF_TMEM_SLOT + 4;
constexpr int kSmemUsed = OFF_ABORT + 4;
constexpr int kSmemBytes = kSmemUsed + 1024;  // + alignment slack

constexpr uint32_t TM_O = 0, TM_S = 256, TM_Q = 384, kTmemCols = 512;
constexpr uint32_t kIdescS = idesc_bf16_f32(128, 64, 0, 0);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 256, 0, 1);
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P stays <= 256
constexpr long long kTimeoutCycles = 2000000000LL;

static_assert(kSmemBytes <= 232448, "shared memory budget");

__device__ int g_kernel_error;

struct Ctx {
  uint8_t* smem;     // 1024-aligned base
  uint32_t sbase;    // its shared-window address
  volatile int* abort_flag;
  __device__ uint32_t bar(int i) const { return sbase + OFF_BAR + 8 * i; }
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

__device__ __forceinline__ int segment_tiles(const Segment& sg, int L) {
  const int last = (L + kTileTokens - 1) / kTileTokens;
  const int e = sg.tile_end < last ? sg.tile_end : last;
  return e > sg.tile_begin ? e - sg.tile_begin : 0;
}

// ------------------------------------------------------------------ producer

template <int CAP>
__device__ void producer(const Ctx& c, const Schedule<CAP>& sched, const DecodeArgs& a, const CUtensorMap* tm_lat,
                         const CUtensorMap* tm_rope, int worker, int rank) {
  const int lane = threadIdx.x & 31;
  const int oob_row = (int)(a.num_pages * a.page_size);  // first row past the pool: zero-filled by TMA
  const int pieces = kTileTokens / a.page_size;           // pages per tile: 1 or 2
  int j = 0, tails = 0;
  bool ok = true;
  for (int s = sched.worker_seg[worker]; ok && s < sched.worker_seg[worker + 1]; ++s) {
    const Segment sg = sched.seg[s];
    const int L = request_len(a, sg.req);
    const int nt = segment_tiles(sg, L);
    const int32_t* bt = a.block_table + (size_t)sg.req * a.bt_stride;
    for (int jj = 0; jj < nt; ++jj, ++j) {
      const int stage = j % kStages;
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
      if (lane == 0) {
        mbar_arrive_expect_tx(land, kStageTx);
        for (int pc = 0; pc < pieces; ++pc) {
          const int ptok = tok0 + pc * a.page_size;
          int y = oob_row;
          if (ptok < L) {
            const int pid = bt[ptok / a.page_size];
            if (pid >= 0 && pid < a.num_pages) y = pid * a.page_size;
          }
          const uint32_t rows = pc * a.page_size;
#pragma unroll
          for (int bx = 0; bx < 4; ++bx)
            tma_load_2d(dst + bx * kLatBox + rows * 128, tm_lat, land, 256 * rank + 64 * bx, y);
          tma_load_2d(dst + 4 * kLatBox + rows * 64, tm_rope, land, 512 + 32 * rank, y);
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
  for (int k = issued - 1; k >= 0 && k >= issued - kStages; --k) {
    const long long t0 = clock64();
    while (!mbar_try_wait(c.bar(B_KV_FULL + (k % kStages)), (k / kStages) & 1) && clock64() - t0 < kTimeoutCycles) {
    }
  }
}

// ------------------------------------------------------------------ MMA issuer

template <int CAP>
__device__ void mma_issuer(const Ctx& c, const Schedule<CAP>& sched, const DecodeArgs& a, uint32_t tmem, int worker) {
  int j = 0, segs_run = 0;
  bool ok = true;
  auto issue_pv = [&](int jp, bool first) -> bool {
    const int pb = jp & 1;
    if (!wait_bar<false>(c, c.bar(B_P_FULL + pb), (jp >> 1) & 1, 0x203)) return false;
    tc_fence_after();
    const uint32_t stage_addr = c.sbase + OFF_KV + (jp % kStages) * kStageBytes;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      // B = V (tokens x 256 latent), MN-major 128B swizzle: 64-column atoms
      // 8 KB apart (LBO), 8-token row groups 1 KB apart (SBO)
      const uint64_t bdesc = smem_desc(stage_addr + kk * 16 * 128, kLatBox, 1024, kSwizzle128B);
      mma_ts(tmem + TM_O, tmem + TM_S + 64 * pb + 8 * kk, bdesc, kIdescPV, (first && kk == 0) ? 0u : 1u);
    }
    mma_commit(c.bar(B_PV_DONE));
    mma_commit(c.bar(B_KV_EMPTY + (jp % kStages)));
    return true;
  };
  for (int s = sched.worker_seg[worker]; ok && s < sched.worker_seg[worker + 1]; ++s) {
    const Segment sg = sched.seg[s];
    const int nt = segment_tiles(sg, request_len(a, sg.req));
    if (nt == 0) continue;
    if (!wait_bar<false>(c, c.bar(B_Q_READY), segs_run & 1, 0x201)) { ok = false; break; }
    ++segs_run;
    tc_fence_after();
    for (int jj = 0; jj < nt; ++jj, ++j) {
      const int stage = j % kStages;
      if (!wait_bar<false>(c, c.bar(B_KV_FULL + stage), (j / kStages) & 1, 0x202)) { ok = false; break; }
      tc_fence_after();
      const uint32_t stage_addr = c.sbase + OFF_KV + stage * kStageBytes;
      const uint32_t d = tmem + TM_S + 64 * (j & 1);
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
      mma_commit(c.bar(B_S_FULL + (j & 1)));
      if (jj > 0 && !issue_pv(j - 1, jj == 1)) { ok = false; break; }
    }
    if (ok && !issue_pv(j - 1, nt == 1)) ok = false;
  }
  // all issued tensor-core work must finish before TMEM is released
  mma_commit(c.bar(B_FINAL));
  const long long t0 = clock64();
  while (!mbar_try_wait(c.bar(B_FINAL), 0) && clock64() - t0 < kTimeoutCycles) {
  }
}

// ------------------------------------------------------------------ softmax

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi, float& rlo, float& rhi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  rlo = __low2float(v);
  rhi = __high2float(v);
  return *reinterpret_cast<uint32_t*>(&v);
}

template <int CAP>
__device__ void softmax_epilogue(const Ctx& c, const Schedule<CAP>& sched, const DecodeArgs& a, uint32_t tmem,
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
  const int qi = valid_row ? row / a.num_heads : 0;  // query position of this row
  // Exchange buffers, [16-byte chunk][row] so a warp's stores are contiguous.
  // This thread's 8 chunks start at chunk 8*half.
  const uint32_t my_off = static_cast<uint32_t>((half * 8 * 128 + row) * 16);
  const uint32_t xchg_local = c.sbase + OFF_XCHG + my_off;
  const uint32_t xchg_peer = mapa(c.sbase + OFF_XCHG, peer) + my_off;
  const uint32_t x_full_peer0 = mapa(c.bar(B_X_FULL), peer), x_full_peer1 = mapa(c.bar(B_X_FULL + 1), peer);
  const uint32_t x_empty_peer0 = mapa(c.bar(B_X_EMPTY), peer), x_empty_peer1 = mapa(c.bar(B_X_EMPTY + 1), peer);
  const uint32_t sink_peer = mapa(c.sbase + OFF_SINK, peer) + (threadIdx.x - 128) * 4;
  float* red_max = reinterpret_cast<float*>(c.smem + OFF_RED);      // [2 tiles][2 halves][128]
  float* red_l = red_max + 2 * 2 * 128;                              // [2 segments][2 halves][128]
  const float cs = a.score_scale_log2;  // raw score -> base-2 logit
  int j = 0, nseg = 0;
  bool ok = true;

  // S partial of tile jn (this thread's 32 columns) from TMEM
  auto load_s = [&](int jn, uint32_t(&sv)[32]) -> bool {
    const int sb = jn & 1;
    if (!wait_bar_warp<false>(c, c.bar(B_S_FULL + sb), (jn >> 1) & 1, 0x301)) return false;
    tc_fence_after();
    tmem_ld32(tmem + lane_off + TM_S + 64 * sb + 32 * half, sv);
    tmem_ld_wait(sv);
    return true;
  };
  // ... and into the peer CTA's exchange buffer
  auto send = [&](int jn, const uint32_t(&sv)[32]) -> bool {
    const int sb = jn & 1, u = jn >> 1;
    if (u > 0 && !wait_bar_warp<true>(c, c.bar(B_X_EMPTY + sb), (u - 1) & 1, 0x302)) return false;
    const uint32_t dst = xchg_peer + sb * kXchgBytes;
    const uint32_t mb = sb ? x_full_peer1 : x_full_peer0;
#pragma unroll
    for (int ch = 0; ch < 8; ++ch)
      st_async_v4(dst + ch * 2048, sv[4 * ch], sv[4 * ch + 1], sv[4 * ch + 2], sv[4 * ch + 3], mb);
    // arm the "peer has read it" phase of this buffer: 256 four-byte notes
    if (threadIdx.x == 128) mbar_arrive_expect_tx(c.bar(B_X_EMPTY + sb), kNoteBytes);
    return true;
  };

  for (int s = sched.worker_seg[worker]; ok && s < sched.worker_seg[worker + 1]; ++s) {
    const Segment sg = sched.seg[s];
    const int b = sg.req;
    const int L = request_len(a, b);
    const int nt = segment_tiles(sg, L);
    const int vis = valid_row ? L - a.q_len + 1 + qi : 0;  // visible keys of this row
    float m_ref = -CUDART_INF_F, l = 0.f;

    if (nt > 0) {
      // ---- Q: latent half -> TMEM columns [384, 512) (this thread: 128 of
      // the 256 elements), rope half -> shared memory (64B swizzle)
      {
        uint32_t r[32];
        const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(a.q_nope) +
                                                          ((size_t)b * M + row) * kLatent + 256 * rank + 128 * half);
#pragma unroll
        for (int ck = 0; ck < 2; ++ck) {
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            const uint4 q4 = valid_row ? __ldg(src + ck * 8 + v) : make_uint4(0, 0, 0, 0);
            r[4 * v + 0] = q4.x; r[4 * v + 1] = q4.y; r[4 * v + 2] = q4.z; r[4 * v + 3] = q4.w;
          }
          tmem_st32(tmem + lane_off + TM_Q + 64 * half + 32 * ck, r);
        }
        const uint4* srp = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(a.q_pe) +
                                                          ((size_t)b * M + row) * kRope + 32 * rank + 16 * half);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int ch = 2 * half + i;
          const uint4 q4 = valid_row ? __ldg(srp + i) : make_uint4(0, 0, 0, 0);
          st_shared_v4(c.sbase + OFF_QROPE + row * 64 + ((ch ^ ((row >> 1) & 3)) << 4), q4);
        }
        tmem_st_wait();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(c.bar(B_Q_READY));
      }

      uint32_t cur[32];  // own partial scores of the tile being finished
      if (!load_s(j, cur) || !send(j, cur)) { ok = false; break; }
      for (int jj = 0; jj < nt; ++jj, ++j) {
        const int sb = j & 1;
        // ---- the next tile's exchange first, so its DSMEM transit overlaps this tile
        uint32_t nxt[32];
        if (jj + 1 < nt && (!load_s(j + 1, nxt) || !send(j + 1, nxt))) { ok = false; break; }
        // ---- full scores: own partial + the peer's (its st.async bytes
        // complete the transaction count this CTA expects per tile)
        if (threadIdx.x == 128) mbar_arrive_expect_tx(c.bar(B_X_FULL + sb), kXchgBytes);
        if (!wait_bar_warp<true>(c, c.bar(B_X_FULL + sb), (j >> 1) & 1, 0x303)) { ok = false; break; }
        float x[32];
        {
          const uint32_t srcx = xchg_local + sb * kXchgBytes;
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            const uint4 v = ld_shared_v4(srcx + ch * 2048);
            x[4 * ch + 0] = __uint_as_float(cur[4 * ch + 0]) + __uint_as_float(v.x);
            x[4 * ch + 1] = __uint_as_float(cur[4 * ch + 1]) + __uint_as_float(v.y);
            x[4 * ch + 2] = __uint_as_float(cur[4 * ch + 2]) + __uint_as_float(v.z);
            x[4 * ch + 3] = __uint_as_float(cur[4 * ch + 3]) + __uint_as_float(v.w);
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
        st_async_b32(sink_peer + sb * kNoteBytes, __float_as_uint(mt), sb ? x_empty_peer1 : x_empty_peer0);
        red_max[(sb * 2 + half) * 128 + row] = mt;
        mbar_arrive(c.bar(B_PAIR_MAX + 2 * quad + sb));
        if (!wait_bar_warp<false>(c, c.bar(B_PAIR_MAX + 2 * quad + sb), (j >> 1) & 1, 0x306)) { ok = false; break; }
        mt = fmaxf(red_max[(sb * 2) * 128 + row], red_max[(sb * 2 + 1) * 128 + row]) * cs;
        // ---- O is idle once the previous tile's P.V is done
        if (jj > 0) {
          if (!wait_bar_warp<false>(c, c.bar(B_PV_DONE), (j - 1) & 1, 0x304)) { ok = false; break; }
          tc_fence_after();
        }
        // lazy rescale: the reference max moves only when it grew by more than
        // 2^8; both halves decide identically; TMEM traffic by whole warps
        const float m_new = fmaxf(m_ref, mt);
        const bool resc = m_new > m_ref + kRescaleThreshold;
        const float alpha = resc ? ex2_approx(m_ref - m_new) : 1.f;  // 0 when m_ref = -inf
        if (jj > 0 && __any_sync(0xffffffffu, resc)) {
#pragma unroll 1
          for (int ck = 0; ck < 4; ++ck) {
            uint32_t o[32];
            const uint32_t addr = tmem + lane_off + TM_O + 128 * half + 32 * ck;
            tmem_ld32(addr, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int v = 0; v < 32; ++v) o[v] = __float_as_uint(__uint_as_float(o[v]) * alpha);
            tmem_st32(addr, o);
          }
          tmem_st_wait();
        }
        if (resc) {
          l *= alpha;
          m_ref = m_new;
        }
        const float nm = m_ref == -CUDART_INF_F ? 0.f : -m_ref;  // all-masked rows: 2^-inf = 0
        // ---- P (bf16 pairs) over the S columns it came from
        uint32_t pk[16];
        float lsum = 0.f;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float p0 = ex2_approx(fmaf(x[2 * k], cs, nm));
          const float p1 = ex2_approx(fmaf(x[2 * k + 1], cs, nm));
          float r0, r1;
          pk[k] = pack_bf16(p0, p1, r0, r1);
          lsum += p0 + p1;  // l from the unrounded probabilities: exact lse
        }
        l += lsum;
        tmem_st16(tmem + lane_off + TM_S + 64 * sb + 16 * half, pk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(c.bar(B_P_FULL + sb));
#pragma unroll
        for (int k = 0; k < 32; ++k) cur[k] = nxt[k];
      }
      if (!ok) break;
      if (!wait_bar_warp<false>(c, c.bar(B_PV_DONE), (j - 1) & 1, 0x305)) { ok = false; break; }
      tc_fence_after();
    }

    // ---- epilogue: row sum over both halves; this thread writes 128 of the
    // CTA's 256 output columns, (rank 0, half 0) the lse.  TMEM is read by
    // whole warps (only when the segment ran MMAs); stores are per row.
    {
      float* rl = red_l + (nseg & 1) * 256;
      rl[half * 128 + row] = l;
      mbar_arrive(c.bar(B_PAIR_L + quad));
      if (!wait_bar_warp<false>(c, c.bar(B_PAIR_L + quad), nseg & 1, 0x307)) { ok = false; break; }
      l = rl[row] + rl[128 + row];
      ++nseg;
    }
    {
      const size_t orow = (size_t)b * M + row;
      const bool live = l > 0.f;
      const float inv = live ? a.out_scale / l : 0.f;
#pragma unroll 1
      for (int ck = 0; ck < 4; ++ck) {
        uint32_t o[32];
        if (nt > 0) {
          tmem_ld32(tmem + lane_off + TM_O + 128 * half + 32 * ck, o);
          tmem_ld_wait(o);
        }
        if (nt == 0 || !live) {
#pragma unroll
          for (int v = 0; v < 32; ++v) o[v] = 0u;
        }
        const int col = 256 * rank + 128 * half + 32 * ck;
        if (!valid_row) continue;
        if (sg.slot < 0) {
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) + orow * kLatent + col);
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
          float4* dst = reinterpret_cast<float4*>(a.part_o + ((size_t)sg.slot * M + row) * kLatent + col);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            dst[v] = make_float4(__uint_as_float(o[4 * v + 0]) * inv, __uint_as_float(o[4 * v + 1]) * inv,
                                 __uint_as_float(o[4 * v + 2]) * inv, __uint_as_float(o[4 * v + 3]) * inv);
        }
      }
      if (rank == 0 && half == 0 && valid_row) {
        const float lse = live ? (m_ref + __log2f(l)) * 0.6931471805599453f : -CUDART_INF_F;
        if (sg.slot < 0) a.lse[orow] = lse;
        else a.part_lse[(size_t)sg.slot * M + row] = lse;
      }
    }
    tc_fence_before();
  }
}

// ------------------------------------------------------------------ kernel

template <int CAP>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ Schedule<CAP> sched, const __grid_constant__ DecodeArgs a,
                  const __grid_constant__ CUtensorMap tm_lat, const __grid_constant__ CUtensorMap tm_rope) {
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

  if (threadIdx.x == 0) {
    *c.abort_flag = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(c.bar(B_KV_FULL + s), 1);
      mbar_init(c.bar(B_KV_EMPTY + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(c.bar(B_S_FULL + i), 1);
      mbar_init(c.bar(B_P_FULL + i), 256);
      mbar_init(c.bar(B_X_FULL + i), 1);  // own expect_tx arrival + the peer's st.async bytes
      mbar_init(c.bar(B_X_EMPTY + i), 1);  // own expect_tx arrival + the peer's 4-byte notes
    }
    mbar_init(c.bar(B_PV_DONE), 1);
    mbar_init(c.bar(B_Q_READY), 256);
    mbar_init(c.bar(B_TAIL), 1);
    mbar_init(c.bar(B_FINAL), 1);
    for (int i = 0; i < 8; ++i) mbar_init(c.bar(B_PAIR_MAX + i), 64);
    for (int i = 0; i < 4; ++i) mbar_init(c.bar(B_PAIR_L + i), 64);
    fence_mbar_init();
    prefetch_tensormap(&tm_lat);
    prefetch_tensormap(&tm_rope);
  }
  if (warp == 1) {
    tmem_alloc(c.sbase + OFF_TMEM_SLOT, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // peer barriers initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(c.smem + OFF_TMEM_SLOT);

  if (worker < sched.num_workers) {
    if (warp == 0) {
      producer<CAP>(c, sched, a, &tm_lat, &tm_rope, worker, rank);
    } else if (warp == 1) {
      if ((threadIdx.x & 31) == 0) mma_issuer<CAP>(c, sched, a, tmem, worker);
      __syncwarp();
    } else if (warp >= 4) {
      softmax_epilogue<CAP>(c, sched, a, tmem, worker, rank);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
  cluster_sync();  // no peer may still write into this CTA's shared memory
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

// 2-D view [num_pages * page_size rows, 576 columns] of the cache.
static bool make_map(CUtensorMap* m, const void* kv, int64_t rows, int box_cols, int box_rows,
                     CUtensorMapSwizzle sw) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kKvDim, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kKvDim * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(kv), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int CAP>
static cudaError_t launch_cap(const mla_plan& p, const DecodeArgs& a, const CUtensorMap& lat,
                              const CUtensorMap& rope, cudaStream_t stream) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(decode_kernel<CAP>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  });
  if (attr_err != cudaSuccess) return attr_err;
  Schedule<CAP> s;
  s.num_workers = p.num_workers;
  s.num_segments = (int32_t)p.segs.size();
  for (int w = 0; w <= p.num_workers; ++w) s.worker_seg[w] = p.worker_seg[w];
  for (size_t i = 0; i < p.segs.size(); ++i) s.seg[i] = p.segs[i];
  decode_kernel<CAP><<<dim3(2 * p.num_workers), kThreads, kSmemBytes, stream>>>(s, a, lat, rope);
  return cudaGetLastError();
}

}  // namespace sm103

// Returns cudaErrorNotSupported when the tensor-map encoder is unavailable.
cudaError_t launch_sm103(const mla_plan& p, const DecodeArgs& a, cudaStream_t stream) {
  CUtensorMap lat, rope;
  const int64_t rows = a.num_pages * a.page_size;
  if (!sm103::make_map(&lat, a.kv, rows, 64, a.page_size, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !sm103::make_map(&rope, a.kv, rows, 32, a.page_size, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorNotSupported;
  if (p.segs.size() <= (size_t)kSegCapSmall) return sm103::launch_cap<kSegCapSmall>(p, a, lat, rope, stream);
  return sm103::launch_cap<kSegCapLarge>(p, a, lat, rope, stream);
}

// Kernel-side error code recorded since the last reset (0 = none).
cudaError_t sm103_read_error(int* code, bool reset) {
  cudaError_t e = cudaMemcpyFromSymbol(code, sm103::g_kernel_error, sizeof(int));
  if (e != cudaSuccess || !reset) return e;
  const int zero = 0;
  return cudaMemcpyToSymbol(sm103::g_kernel_error, &zero, sizeof(int));
}

}  // namespace mla
