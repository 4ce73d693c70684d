// The step that feeds the decode: rotary embedding of the rope parts, FP8
// (e4m3) quantisation, and the write of each new token's latent row into
// the paged cache -- one launch for the query and the key (sglang
// trtllm_mla_backend.py, forward_decode: mla_quantize_and_rope_for_fp8, then
// set_mla_kv_buffer(out_cache_loc, k, k_rope); tokenspeed trtllm_mla.py,
// forward_decode: set_mla_kv_buffer).
//
// Work item = 8 elements of one row: a chunk of the 512 latent columns, or 4
// rotated pairs of the 64 rope columns; a token has (num_heads + 1) rows of
// 72 items (its query heads, then its key).  One thread per item: the loads
// are 16-byte (8-byte for a half-split rope chunk), the stores 8 or 16
// bytes.  Memory bound: per token 1152 B read per head and per key,
// 576 (e4m3) or 1152 (bf16) bytes written per output row.
//
// Rotation: pair (a, b) -> (a cos - b sin, b cos + a sin) in fp32 (each
// product and sum rounded on its own), with
// cos/sin from cos_sin_cache[position] ([32 cos | 32 sin] fp32); the pairs
// are (i, i + 32) when is_neox, else (2i, 2i + 1).  Quantisation: cvt.rn
// .satfinite.e4m3x2.f32 (nearest even, saturating at 448).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mla_decode.h"

namespace mla_kw {

__device__ int g_kw_error;

constexpr int kThreads = 256;
constexpr int kItemsPerRow = 72;  // 64 latent chunks + 8 rope chunks

__device__ __forceinline__ void record(int code) { atomicCAS(&g_kw_error, 0, code); }

// two floats -> two e4m3 bytes, `lo` at the lower address
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}

__device__ __forceinline__ uint32_t bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

struct Args {
  const uint16_t* q_nope;   // bf16 [T, H, 512]
  const uint16_t* q_rope;   // bf16 [T, H, 64]
  void* q_out;              // e4m3 [T, H, 576] or bf16 [T, H, 64]
  const uint16_t* k_nope;   // bf16 [T, 512]
  const uint16_t* k_rope;   // bf16 [T, 64]
  const int64_t* positions;
  const float* cos_sin;     // [max_position, 64] or nullptr (no rotation)
  void* kv;                 // [P, page, 576] bf16 or e4m3
  const int64_t* slots;
  int64_t max_position;
  int64_t num_slots;        // P * page
  int num_tokens, num_heads, q_e4m3, kv_e4m3, is_neox;
};

// The raw bits of 4 rope pairs (4r .. 4r + 3) of a 64-wide bf16 row: for
// is_neox the 8 bytes of elements 4r.. and the 8 bytes of elements 32 + 4r..,
// otherwise the 16 bytes of elements 8r..
__device__ __forceinline__ uint4 load_pairs_raw(const uint16_t* row, int r, bool neox) {
  if (neox) {
    const uint2 x = *reinterpret_cast<const uint2*>(row + 4 * r);
    const uint2 y = *reinterpret_cast<const uint2*>(row + 32 + 4 * r);
    return make_uint4(x.x, x.y, y.x, y.y);
  }
  return *reinterpret_cast<const uint4*>(row + 8 * r);
}

// ... and as floats: a[k], b[k] are the two elements of pair 4r + k.
__device__ __forceinline__ void unpack_pairs(uint4 v, bool neox, float a[4], float b[4]) {
  if (neox) {
    a[0] = bf_lo(v.x); a[1] = bf_hi(v.x); a[2] = bf_lo(v.y); a[3] = bf_hi(v.y);
    b[0] = bf_lo(v.z); b[1] = bf_hi(v.z); b[2] = bf_lo(v.w); b[3] = bf_hi(v.w);
  } else {
    a[0] = bf_lo(v.x); b[0] = bf_hi(v.x); a[1] = bf_lo(v.y); b[1] = bf_hi(v.y);
    a[2] = bf_lo(v.z); b[2] = bf_hi(v.z); a[3] = bf_lo(v.w); b[3] = bf_hi(v.w);
  }
}

// Store 4 rotated pairs into a 64-wide rope row (e4m3 bytes or bf16).
__device__ __forceinline__ void store_pairs(void* row, bool e4m3, int r, bool neox, const float a[4], const float b[4]) {
  if (e4m3) {
    uint8_t* o = static_cast<uint8_t*>(row);
    if (neox) {
      *reinterpret_cast<uint32_t*>(o + 4 * r) = e4m3x2(a[0], a[1]) | (uint32_t)e4m3x2(a[2], a[3]) << 16;
      *reinterpret_cast<uint32_t*>(o + 32 + 4 * r) = e4m3x2(b[0], b[1]) | (uint32_t)e4m3x2(b[2], b[3]) << 16;
    } else {
      *reinterpret_cast<uint2*>(o + 8 * r) =
          make_uint2(e4m3x2(a[0], b[0]) | (uint32_t)e4m3x2(a[1], b[1]) << 16,
                     e4m3x2(a[2], b[2]) | (uint32_t)e4m3x2(a[3], b[3]) << 16);
    }
  } else {
    uint16_t* o = static_cast<uint16_t*>(row);
    if (neox) {
      *reinterpret_cast<uint2*>(o + 4 * r) = make_uint2(bf16x2(a[0], a[1]), bf16x2(a[2], a[3]));
      *reinterpret_cast<uint2*>(o + 32 + 4 * r) = make_uint2(bf16x2(b[0], b[1]), bf16x2(b[2], b[3]));
    } else {
      *reinterpret_cast<uint4*>(o + 8 * r) =
          make_uint4(bf16x2(a[0], b[0]), bf16x2(a[1], b[1]), bf16x2(a[2], b[2]), bf16x2(a[3], b[3]));
    }
  }
}

// 8 latent values (one 16-byte chunk of a bf16 row) into e4m3 or bf16.
__device__ __forceinline__ void store_latent(void* dst, bool e4m3, uint4 x) {
  if (e4m3) {
    *reinterpret_cast<uint2*>(dst) =
        make_uint2(e4m3x2(bf_lo(x.x), bf_hi(x.x)) | (uint32_t)e4m3x2(bf_lo(x.y), bf_hi(x.y)) << 16,
                   e4m3x2(bf_lo(x.z), bf_hi(x.z)) | (uint32_t)e4m3x2(bf_lo(x.w), bf_hi(x.w)) << 16);
  } else {
    *reinterpret_cast<uint4*>(dst) = x;  // bf16 -> bf16: the stored bits
  }
}

// (a, b) -> (a c - b s, b c + a s), each product and the sum rounded to fp32
// on its own (no fused multiply-add), so the value a code is rounded from is
// fixed by the formula alone.
__device__ __forceinline__ void rotate4(const float x[4], const float y[4], const float c[4], const float s[4],
                                        float ra[4], float rb[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    ra[i] = __fsub_rn(__fmul_rn(x[i], c[i]), __fmul_rn(y[i], s[i]));
    rb[i] = __fadd_rn(__fmul_rn(y[i], c[i]), __fmul_rn(x[i], s[i]));
  }
}

// One thread per item over a flat grid.  Each thread issues its independent
// loads -- the position, the slot and the source chunk -- before anything
// that depends on them, then the cos / sin pair the position selects: two
// memory round trips in all.
__global__ void __launch_bounds__(kThreads) rope_quantize_write_kernel(const Args a) {
  const int64_t item = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  const int per_token = (a.num_heads + 1) * kItemsPerRow;
  if (item >= (int64_t)per_token * a.num_tokens) return;
  const int t = (int)(item / per_token);
  const int rem = (int)(item - (int64_t)t * per_token);
  const int h = rem / kItemsPerRow;  // h == num_heads: the key row
  const int w = rem - h * kItemsPerRow;
  const bool is_key = h == a.num_heads;
  // ---- independent loads
  const int64_t pos = a.cos_sin ? a.positions[t] : 0;
  const int64_t slot = is_key ? a.slots[t] : 0;
  const int64_t qrow = (int64_t)t * a.num_heads + h;
  uint4 x = make_uint4(0u, 0u, 0u, 0u);
  if (w < 64) {
    if (is_key)
      x = *reinterpret_cast<const uint4*>(a.k_nope + (int64_t)t * 512 + 8 * w);
    else if (a.q_e4m3)
      x = *reinterpret_cast<const uint4*>(a.q_nope + qrow * 512 + 8 * w);
  } else {
    x = load_pairs_raw(is_key ? a.k_rope + (int64_t)t * 64 : a.q_rope + qrow * 64, w - 64, a.is_neox);
  }
  if (a.cos_sin && (pos < 0 || pos >= a.max_position)) {
    if (w == 64 && (is_key || h == 0)) record(0x601);
    return;  // nothing of this token is written
  }
  // ---- rotation of the rope chunks (identity without a cos/sin table)
  float ra[4], rb[4];
  if (w >= 64) {
    float c[4] = {1.f, 1.f, 1.f, 1.f}, sn[4] = {0.f, 0.f, 0.f, 0.f};
    if (a.cos_sin) {
      const int r = w - 64;
      const float4 cv = *reinterpret_cast<const float4*>(a.cos_sin + pos * 64 + 4 * r);
      const float4 sv = *reinterpret_cast<const float4*>(a.cos_sin + pos * 64 + 32 + 4 * r);
      c[0] = cv.x; c[1] = cv.y; c[2] = cv.z; c[3] = cv.w;
      sn[0] = sv.x; sn[1] = sv.y; sn[2] = sv.z; sn[3] = sv.w;
    }
    float xa[4], xb[4];
    unpack_pairs(x, a.is_neox, xa, xb);
    rotate4(xa, xb, c, sn, ra, rb);
  }
  // ---- stores
  if (is_key) {
    if (slot < 0 || slot >= a.num_slots) {
      if (w == 0) record(0x602);
      return;
    }
    uint8_t* row = static_cast<uint8_t*>(a.kv) + slot * (a.kv_e4m3 ? 576 : 1152);
    if (w < 64)
      store_latent(row + (a.kv_e4m3 ? 8 : 16) * w, a.kv_e4m3, x);
    else
      store_pairs(row + (a.kv_e4m3 ? 512 : 1024), a.kv_e4m3, w - 64, a.is_neox, ra, rb);
  } else if (w < 64) {
    if (a.q_e4m3)  // a bf16 query's latent part is used as it is
      store_latent(static_cast<uint8_t*>(a.q_out) + qrow * 576 + 8 * w, true, x);
  } else {
    void* dst = a.q_e4m3 ? static_cast<void*>(static_cast<uint8_t*>(a.q_out) + qrow * 576 + 512)
                         : static_cast<void*>(static_cast<uint16_t*>(a.q_out) + qrow * 64);
    store_pairs(dst, a.q_e4m3, w - 64, a.is_neox, ra, rb);
  }
}

}  // namespace mla_kw

namespace mla {

cudaError_t launch_rope_quantize_write(const void* q_nope, const void* q_rope, int num_tokens, int num_heads,
                                       void* q_out, int q_out_dtype, const void* k_nope, const void* k_rope,
                                       const int64_t* positions, const float* cos_sin_cache, int64_t max_position,
                                       int is_neox, void* kv_pages, int kv_dtype, int64_t num_pages, int page_size,
                                       const int64_t* out_cache_loc, cudaStream_t stream) {
  mla_kw::Args a;
  a.q_nope = static_cast<const uint16_t*>(q_nope);
  a.q_rope = static_cast<const uint16_t*>(q_rope);
  a.q_out = q_out;
  a.k_nope = static_cast<const uint16_t*>(k_nope);
  a.k_rope = static_cast<const uint16_t*>(k_rope);
  a.positions = positions;
  a.cos_sin = cos_sin_cache;
  a.kv = kv_pages;
  a.slots = out_cache_loc;
  a.max_position = max_position;
  a.num_slots = num_pages * page_size;
  a.num_tokens = num_tokens;
  a.num_heads = num_heads;
  a.q_e4m3 = q_out_dtype == MLA_Q_E4M3;
  a.kv_e4m3 = kv_dtype == MLA_KV_E4M3;
  a.is_neox = is_neox != 0;
  const int64_t items = (int64_t)num_tokens * (num_heads + 1) * mla_kw::kItemsPerRow;
  const unsigned blocks = (unsigned)((items + mla_kw::kThreads - 1) / mla_kw::kThreads);
  mla_kw::rope_quantize_write_kernel<<<blocks, mla_kw::kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t kv_write_read_error(int* code, bool reset) {
  cudaError_t e = cudaMemcpyFromSymbol(code, mla_kw::g_kw_error, sizeof(int));
  if (e != cudaSuccess || !reset) return e;
  const int zero = 0;
  return cudaMemcpyToSymbol(mla_kw::g_kw_error, &zero, sizeof(int));
}

}  // namespace mla
