// Block-table construction: the step the serving pages run right before the
// decode, turning a request pool into the [batch, max_blocks] page list the
// decode reads (sglang trtllm_mla_backend.py, _create_block_kv_indices and
// create_flashmla_kv_indices_triton; tokenspeed trtllm_mla.py,
// _create_block_kv_indices; tokenspeed flashmla.py, _init_decode_metadata).
//
// Both variants are pure gathers of a few KB, bound by launch latency rather
// than by HBM: one thread per table entry, a 2-D grid (request, 256-entry
// chunk) so a request's pool row and length are read once per CTA and the
// table writes are coalesced.  Lookups outside the pool write the padding
// value and record an error code instead of reading out of bounds.
#include <cuda_runtime.h>
#include <stdint.h>

namespace mla_bt {

__device__ int g_bt_error;

constexpr int kThreads = 256;

__device__ __forceinline__ void record(int code) { atomicCAS(&g_bt_error, 0, code); }

// Entry i < ceil(L / page) of request b: the page holding the slot of the
// first token of its page i (slot = page id * page_size + offset); -1 after.
__global__ void __launch_bounds__(kThreads) from_tokens_kernel(
    const int32_t* __restrict__ req_to_token, int64_t pool_rows, int64_t token_cols,
    const int32_t* __restrict__ req_pool_indices, const int32_t* __restrict__ seq_lens,
    int page_shift, int32_t* __restrict__ block_table, int max_blocks) {
  const int b = blockIdx.x;
  const int i = blockIdx.y * kThreads + threadIdx.x;
  if (i >= max_blocks) return;
  const int L = __ldg(seq_lens + b);
  const int64_t row = __ldg(req_pool_indices + b);
  int32_t v = -1;
  if (L < 0) {
    if (i == 0) record(0x303);
  } else if (i < ((int64_t)L + (1 << page_shift) - 1) >> page_shift) {
    const int64_t col = (int64_t)i << page_shift;
    if (row < 0 || row >= pool_rows) {
      if (i == 0) record(0x301);
    } else if (col >= token_cols) {
      record(0x302);
    } else {
      const int32_t slot = __ldg(req_to_token + row * token_cols + col);
      if (slot < 0)
        record(0x304);
      else
        v = slot >> page_shift;
    }
  }
  block_table[(int64_t)b * max_blocks + i] = v;
}

// Entry i < min(max_blocks, page_cols) of request b: column i of its pool
// row; 0 after.
__global__ void __launch_bounds__(kThreads) from_pages_kernel(
    const int32_t* __restrict__ req_to_page, int64_t pool_rows, int64_t page_cols,
    const int32_t* __restrict__ req_pool_indices, int32_t* __restrict__ block_table, int max_blocks) {
  const int b = blockIdx.x;
  const int i = blockIdx.y * kThreads + threadIdx.x;
  if (i >= max_blocks) return;
  const int64_t row = __ldg(req_pool_indices + b);
  int32_t v = 0;
  if (i < page_cols) {
    if (row < 0 || row >= pool_rows) {
      if (i == 0) record(0x301);
    } else {
      v = __ldg(req_to_page + row * page_cols + i);
    }
  }
  block_table[(int64_t)b * max_blocks + i] = v;
}

}  // namespace mla_bt

namespace mla {

cudaError_t launch_block_table_from_tokens(const int32_t* req_to_token, int64_t pool_rows,
                                           int64_t token_cols, const int32_t* req_pool_indices,
                                           const int32_t* seq_lens, int batch, int page_size,
                                           int32_t* block_table, int max_blocks, cudaStream_t stream) {
  const int shift = page_size == 32 ? 5 : 6;
  dim3 grid(batch, (max_blocks + mla_bt::kThreads - 1) / mla_bt::kThreads);
  mla_bt::from_tokens_kernel<<<grid, mla_bt::kThreads, 0, stream>>>(
      req_to_token, pool_rows, token_cols, req_pool_indices, seq_lens, shift, block_table, max_blocks);
  return cudaGetLastError();
}

cudaError_t launch_block_table_from_pages(const int32_t* req_to_page, int64_t pool_rows, int64_t page_cols,
                                          const int32_t* req_pool_indices, int batch, int32_t* block_table,
                                          int max_blocks, cudaStream_t stream) {
  dim3 grid(batch, (max_blocks + mla_bt::kThreads - 1) / mla_bt::kThreads);
  mla_bt::from_pages_kernel<<<grid, mla_bt::kThreads, 0, stream>>>(req_to_page, pool_rows, page_cols,
                                                                   req_pool_indices, block_table, max_blocks);
  return cudaGetLastError();
}

cudaError_t block_table_read_error(int* code, bool reset) {
  cudaError_t e = cudaMemcpyFromSymbol(code, mla_bt::g_bt_error, sizeof(int));
  if (e != cudaSuccess || !reset) return e;
  const int zero = 0;
  return cudaMemcpyToSymbol(mla_bt::g_bt_error, &zero, sizeof(int));
}

}  // namespace mla
