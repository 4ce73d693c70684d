// C ABI shim: argument validation, plan handling and kernel launches.
// Every argument error is caught here, on the host, before any launch.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <string>

#include "../../include/mla_decode.h"
#include "mla_internal.h"

namespace mla {
cudaError_t launch_sm103(const mla_plan& p, const DecodeArgs& a, const void* workspace, cudaStream_t stream);
cudaError_t launch_plan_device(const int32_t* seq_lens, int batch, int cap_tokens, int workers, void* workspace,
                               cudaStream_t stream);
cudaError_t launch_combine_dev(int workers, const DecodeArgs& a, const void* workspace, cudaStream_t stream);
cudaError_t sm103_read_error(int* code, bool reset);
cudaError_t launch_combine(const std::vector<CombineJob>& jobs, const DecodeArgs& a,
                           cudaStream_t stream);
cudaError_t launch_block_table_from_tokens(const int32_t* req_to_token, int64_t pool_rows,
                                           int64_t token_cols, const int32_t* req_pool_indices,
                                           const int32_t* seq_lens, int batch, int page_size,
                                           int32_t* block_table, int max_blocks, cudaStream_t stream);
cudaError_t launch_block_table_from_pages(const int32_t* req_to_page, int64_t pool_rows, int64_t page_cols,
                                          const int32_t* req_pool_indices, int batch, int32_t* block_table,
                                          int max_blocks, cudaStream_t stream);
cudaError_t block_table_read_error(int* code, bool reset);
cudaError_t launch_rope_quantize_write(const void* q_nope, const void* q_rope, int num_tokens, int num_heads,
                                       void* q_out, int q_out_dtype, const void* k_nope, const void* k_rope,
                                       const int64_t* positions, const float* cos_sin_cache, int64_t max_position,
                                       int is_neox, void* kv_pages, int kv_dtype, int64_t num_pages, int page_size,
                                       const int64_t* out_cache_loc, cudaStream_t stream);
cudaError_t kv_write_read_error(int* code, bool reset);
}  // namespace mla

namespace {

thread_local std::string g_last_error;

int fail(int code, const std::string& msg) {
  g_last_error = msg;
  return code;
}

int ok() {
  g_last_error.clear();
  return MLA_OK;
}

// Per-device capability cache: 1 = sm_103, -1 = other, 0 = unknown.
int g_dev_ok[64];
int g_dev_sms[64];
std::mutex g_dev_mu;

int check_device(int* sms_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return fail(MLA_ERR_UNSUPPORTED, "device index out of range");
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (g_dev_ok[dev] == 0) {
    int maj = 0, min = 0, sms = 0;
    if (cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&min, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return fail(MLA_ERR_CUDA, "cudaDeviceGetAttribute failed");
    g_dev_ok[dev] = (maj == 10 && min == 3) ? 1 : -1;
    g_dev_sms[dev] = sms;
  }
  if (g_dev_ok[dev] != 1)
    return fail(MLA_ERR_UNSUPPORTED, "this library holds sm_103a code only (GB300 class GPU required)");
  if (sms_out) *sms_out = g_dev_sms[dev];
  return MLA_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Prepared {
  mla::DecodeArgs args;
  void* workspace = nullptr;
};

// cu_seqlens_q: NULL for a uniform batch (num_tokens = batch * q_len), else
// the ragged query offsets (1 <= num_tokens <= batch * planned maximum).
int prepare(const mla_plan* plan, const void* q_nope, const void* q_pe, int num_tokens, int num_heads,
            const void* kv_pages, int kv_dtype, int64_t num_pages, int page_size,
            const int32_t* block_table, int bt_stride, const int32_t* seq_lens, const int32_t* cu_seqlens_q,
            float scale, float k_scale, void* out, float* lse, void* workspace, size_t workspace_bytes,
            Prepared* pr) {
  if (!plan) return fail(MLA_ERR_ARG, "plan is NULL");
  if (!q_nope || !q_pe || !kv_pages || !block_table || !seq_lens || !out || !lse)
    return fail(MLA_ERR_ARG, "a required device pointer is NULL");
  const bool tokens_ok = cu_seqlens_q ? (num_tokens >= 1 && num_tokens <= plan->batch * plan->q_len)
                                      : num_tokens == plan->batch * plan->q_len;
  if (!tokens_ok || num_heads != plan->num_heads || page_size != plan->page_size)
    return fail(MLA_ERR_PLAN_MISMATCH,
                "num_tokens / num_heads / page_size differ from the plan (re-plan for this batch)");
  if (cu_seqlens_q && !aligned(cu_seqlens_q, 4)) return fail(MLA_ERR_ARG, "cu_seqlens_q must be 4-byte aligned");
  if ((int64_t)num_tokens * num_heads > INT32_MAX) return fail(MLA_ERR_ARG, "num_tokens * num_heads must be < 2^31");
  if (kv_dtype != MLA_KV_BF16 && kv_dtype != MLA_KV_E4M3) return fail(MLA_ERR_ARG, "kv_dtype must be MLA_KV_BF16 or MLA_KV_E4M3");
  if (num_pages <= 0) return fail(MLA_ERR_ARG, "num_pages must be > 0");
  if (num_pages * (int64_t)page_size > INT32_MAX) return fail(MLA_ERR_ARG, "num_pages * page_size must be < 2^31");
  if (bt_stride < 1 || bt_stride < plan->max_pages)
    return fail(MLA_ERR_ARG, "bt_stride is smaller than the pages of the longest planned request");
  if ((int64_t)bt_stride * page_size > INT32_MAX) return fail(MLA_ERR_ARG, "bt_stride * page_size must be < 2^31");
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(MLA_ERR_ARG, "scale must be finite and > 0");
  if (kv_dtype == MLA_KV_E4M3 && (!(k_scale > 0.f) || !std::isfinite(k_scale)))
    return fail(MLA_ERR_ARG, "k_scale must be finite and > 0");
  if (!aligned(kv_pages, 16) || !aligned(q_nope, 16) || !aligned(q_pe, 16) || !aligned(out, 16) ||
      !aligned(lse, 4))
    return fail(MLA_ERR_ARG, "q_nope, q_pe, kv_pages and out must be 16-byte aligned");
  if (plan->ws_bytes > 0) {
    if (!workspace || workspace_bytes < plan->ws_bytes)
      return fail(MLA_ERR_WORKSPACE, "workspace is smaller than mla_plan_workspace_bytes(plan)");
    if (!aligned(workspace, 256)) return fail(MLA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  }
  const float kf = kv_dtype == MLA_KV_E4M3 ? k_scale : 1.0f;  // ignored for a bf16 cache
  mla::DecodeArgs& a = pr->args;
  a.q_nope = q_nope; a.q_pe = q_pe; a.kv = kv_pages;
  a.block_table = block_table; a.seq_lens = seq_lens;
  a.out = out; a.lse = lse;
  a.part_o = workspace ? static_cast<char*>(workspace) + plan->ws_part_offset : nullptr;
  a.part_lse = workspace ? reinterpret_cast<float*>(static_cast<char*>(workspace) + plan->ws_lse_offset) : nullptr;
  pr->workspace = workspace;
  a.num_pages = num_pages; a.page_size = page_size; a.kv_dtype = kv_dtype; a.bt_stride = bt_stride;
  a.batch = plan->batch; a.q_len = plan->q_len; a.num_heads = plan->num_heads; a.rows = plan->rows;
  a.score_scale_log2 = (float)((double)scale * (double)kf * 1.4426950408889634);
  a.out_scale = kf;
  a.cu_q = cu_seqlens_q;
  a.num_tokens = num_tokens;
  a.q_e4m3 = 0;
  return MLA_OK;
}

int launch_main(const mla_plan* plan, const Prepared& pr, cudaStream_t stream) {
  if (plan->device) {
    // the schedule for the lengths now on the device, into the workspace head
    const mla::DecodeArgs& a = pr.args;
    cudaError_t e = mla::launch_plan_device(a.seq_lens, a.batch, a.bt_stride * a.page_size, plan->num_workers,
                                            pr.workspace, stream);
    if (e != cudaSuccess) return fail(MLA_ERR_CUDA, std::string("planner launch: ") + cudaGetErrorString(e));
  }
  cudaError_t e = mla::launch_sm103(*plan, pr.args, pr.workspace, stream);
  if (e == cudaErrorNotSupported)
    return fail(MLA_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled unavailable or rejected the cache layout");
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, std::string("main kernel launch: ") + cudaGetErrorString(e));
  return MLA_OK;
}

int launch_combine(const mla_plan* plan, const Prepared& pr, cudaStream_t stream) {
  cudaError_t e = plan->device ? mla::launch_combine_dev(plan->num_workers, pr.args, pr.workspace, stream)
                               : mla::launch_combine(plan->jobs, pr.args, stream);
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, std::string("combine launch: ") + cudaGetErrorString(e));
  return MLA_OK;
}

}  // namespace

namespace mla {
// Lets other translation units of the library record a failure message.
int report_error(int code, const char* msg) { return fail(code, msg); }
// The device check every entry point makes (sm_103 only), for other
// translation units.
int require_sm103() { return check_device(nullptr); }
}  // namespace mla

extern "C" {

int mla_decode_plan(const int32_t* seq_lens_host, int batch, int page_size, int num_heads, int q_len,
                    int num_sms, mla_plan** plan_out, size_t* workspace_bytes_out) {
  if (!plan_out) return fail(MLA_ERR_ARG, "plan_out is NULL");
  *plan_out = nullptr;
  if (num_sms < 0) return fail(MLA_ERR_ARG, "num_sms must be >= 0");
  if (num_sms == 0) {
    int rc = check_device(&num_sms);
    if (rc != MLA_OK) return rc;
  }
  mla_plan* p = new (std::nothrow) mla_plan();
  if (!p) return fail(MLA_ERR_ARG, "out of host memory");
  const char* msg = "";
  int rc = mla::build_plan(seq_lens_host, batch, page_size, num_heads, q_len, num_sms, p, &msg);
  if (rc != MLA_OK) { delete p; return fail(rc, msg); }
  if (p->segs.size() > (size_t)mla::kSegCapLarge || p->jobs.size() > (size_t)mla::kJobCap) {
    delete p;
    return fail(MLA_ERR_ARG, "batch too large: the schedule exceeds one launch's segment capacity");
  }
  *plan_out = p;
  if (workspace_bytes_out) *workspace_bytes_out = p->ws_bytes;
  return ok();
}

void mla_plan_destroy(mla_plan* plan) { delete plan; }

int mla_decode_main(const mla_plan* plan, const void* q_nope, const void* q_pe, int num_tokens, int num_heads,
                    const void* kv_pages, int kv_dtype, int64_t num_pages, int page_size,
                    const int32_t* block_table, int bt_stride, const int32_t* seq_lens, float scale,
                    float k_scale, void* out, float* lse, void* workspace, size_t workspace_bytes,
                    void* stream) {
  Prepared pr;
  int rc = prepare(plan, q_nope, q_pe, num_tokens, num_heads, kv_pages, kv_dtype, num_pages, page_size,
                   block_table, bt_stride, seq_lens, nullptr, scale, k_scale, out, lse, workspace, workspace_bytes,
                   &pr);
  if (rc != MLA_OK) return rc;
  rc = check_device(nullptr);
  if (rc != MLA_OK) return rc;
  rc = launch_main(plan, pr, static_cast<cudaStream_t>(stream));
  return rc == MLA_OK ? ok() : rc;
}

int mla_decode_combine(const mla_plan* plan, void* out, float* lse, void* workspace, size_t workspace_bytes,
                       void* stream) {
  if (!plan) return fail(MLA_ERR_ARG, "plan is NULL");
  if (plan->jobs.empty() && !plan->device) return ok();
  if (!out || !lse) return fail(MLA_ERR_ARG, "out / lse is NULL");
  if (!workspace || workspace_bytes < plan->ws_bytes)
    return fail(MLA_ERR_WORKSPACE, "workspace is smaller than mla_plan_workspace_bytes(plan)");
  if (!aligned(workspace, 256)) return fail(MLA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  int rc = check_device(nullptr);
  if (rc != MLA_OK) return rc;
  Prepared pr;
  std::memset(&pr, 0, sizeof(pr));
  mla::DecodeArgs& a = pr.args;
  a.out = out; a.lse = lse;
  a.part_o = static_cast<char*>(workspace) + plan->ws_part_offset;
  a.part_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) + plan->ws_lse_offset);
  pr.workspace = workspace;
  a.batch = plan->batch; a.q_len = plan->q_len; a.num_heads = plan->num_heads; a.rows = plan->rows;
  rc = launch_combine(plan, pr, static_cast<cudaStream_t>(stream));
  return rc == MLA_OK ? ok() : rc;
}

int mla_decode(const mla_plan* plan, const void* q_nope, const void* q_pe, int num_tokens, int num_heads,
               const void* kv_pages, int kv_dtype, int64_t num_pages, int page_size, const int32_t* block_table,
               int bt_stride, const int32_t* seq_lens, float scale, float k_scale, void* out, float* lse,
               void* workspace, size_t workspace_bytes, void* stream) {
  Prepared pr;
  int rc = prepare(plan, q_nope, q_pe, num_tokens, num_heads, kv_pages, kv_dtype, num_pages, page_size,
                   block_table, bt_stride, seq_lens, nullptr, scale, k_scale, out, lse, workspace, workspace_bytes,
                   &pr);
  if (rc != MLA_OK) return rc;
  rc = check_device(nullptr);
  if (rc != MLA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  rc = launch_main(plan, pr, s);
  if (rc != MLA_OK) return rc;
  rc = launch_combine(plan, pr, s);
  return rc == MLA_OK ? ok() : rc;
}

int mla_decode_host_io(const mla_plan* plan, void* q_nope, void* q_pe, int num_tokens, int num_heads,
                       const void* kv_pages, int kv_dtype, int64_t num_pages, int page_size,
                       int32_t* block_table, int bt_stride, int32_t* seq_lens, float scale, float k_scale,
                       void* out, float* lse, void* workspace, size_t workspace_bytes,
                       const void* q_nope_host, const void* q_pe_host, const int32_t* block_table_host,
                       const int32_t* seq_lens_host, void* out_host, float* lse_host, void* stream) {
  if (!q_nope_host || !q_pe_host || !block_table_host || !seq_lens_host || !out_host || !lse_host)
    return fail(MLA_ERR_ARG, "a host pointer is NULL");
  Prepared pr;
  int rc = prepare(plan, q_nope, q_pe, num_tokens, num_heads, kv_pages, kv_dtype, num_pages, page_size,
                   block_table, bt_stride, seq_lens, nullptr, scale, k_scale, out, lse, workspace, workspace_bytes,
                   &pr);
  if (rc != MLA_OK) return rc;
  rc = check_device(nullptr);
  if (rc != MLA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t rows = (size_t)num_tokens * num_heads;
  const size_t batch = (size_t)plan->batch;
  struct Copy { void* dst; const void* src; size_t bytes; };
  const Copy in[4] = {{q_nope, q_nope_host, rows * mla::kLatent * 2},
                      {q_pe, q_pe_host, rows * mla::kRope * 2},
                      {block_table, block_table_host, batch * (size_t)bt_stride * 4},
                      {seq_lens, seq_lens_host, batch * 4}};
  for (const Copy& cp : in) {
    const cudaError_t e = cudaMemcpyAsync(cp.dst, cp.src, cp.bytes, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return fail(MLA_ERR_CUDA, std::string("input copy: ") + cudaGetErrorString(e));
  }
  rc = launch_main(plan, pr, s);
  if (rc != MLA_OK) return rc;
  rc = launch_combine(plan, pr, s);
  if (rc != MLA_OK) return rc;
  const Copy res[2] = {{out_host, out, rows * mla::kLatent * 2}, {lse_host, lse, rows * 4}};
  for (const Copy& cp : res) {
    const cudaError_t e = cudaMemcpyAsync(cp.dst, cp.src, cp.bytes, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return fail(MLA_ERR_CUDA, std::string("result copy: ") + cudaGetErrorString(e));
  }
  return ok();
}

int mla_decode_plan_ragged(const int32_t* seq_lens_host, const int32_t* q_lens_host, int batch, int page_size,
                           int num_heads, int num_sms, mla_plan** plan_out, size_t* workspace_bytes_out) {
  if (!plan_out) return fail(MLA_ERR_ARG, "plan_out is NULL");
  *plan_out = nullptr;
  if (!q_lens_host) return fail(MLA_ERR_ARG, "q_lens_host is NULL");
  if (batch < 1) return fail(MLA_ERR_ARG, "batch must be >= 1");
  int q_max = 1;
  for (int b = 0; b < batch; ++b) {
    if (q_lens_host[b] < 0) return fail(MLA_ERR_ARG, "q_lens must be >= 0");
    q_max = std::max(q_max, (int)q_lens_host[b]);
  }
  int rc = mla_decode_plan(seq_lens_host, batch, page_size, num_heads, q_max, num_sms, plan_out,
                           workspace_bytes_out);
  if (rc != MLA_OK) return rc;
  (*plan_out)->ragged = true;
  return ok();
}

int mla_decode_ragged(const mla_plan* plan, const void* q_nope, const void* q_pe, int num_tokens, int num_heads,
                      const void* kv_pages, int kv_dtype, int64_t num_pages, int page_size,
                      const int32_t* block_table, int bt_stride, const int32_t* seq_lens,
                      const int32_t* cu_seqlens_q, float scale, float k_scale, void* out, float* lse,
                      void* workspace, size_t workspace_bytes, void* stream) {
  if (!cu_seqlens_q) return fail(MLA_ERR_ARG, "cu_seqlens_q is NULL");
  Prepared pr;
  int rc = prepare(plan, q_nope, q_pe, num_tokens, num_heads, kv_pages, kv_dtype, num_pages, page_size,
                   block_table, bt_stride, seq_lens, cu_seqlens_q, scale, k_scale, out, lse, workspace,
                   workspace_bytes, &pr);
  if (rc != MLA_OK) return rc;
  rc = check_device(nullptr);
  if (rc != MLA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  rc = launch_main(plan, pr, s);
  if (rc != MLA_OK) return rc;
  rc = launch_combine(plan, pr, s);
  return rc == MLA_OK ? ok() : rc;
}

int mla_decode_plan_device(int batch, int page_size, int num_heads, int q_len, int num_sms, mla_plan** plan_out,
                           size_t* workspace_bytes_out) {
  if (!plan_out) return fail(MLA_ERR_ARG, "plan_out is NULL");
  *plan_out = nullptr;
  if (num_sms < 0) return fail(MLA_ERR_ARG, "num_sms must be >= 0");
  if (num_sms == 0) {
    int rc = check_device(&num_sms);
    if (rc != MLA_OK) return rc;
  }
  mla_plan* p = new (std::nothrow) mla_plan();
  if (!p) return fail(MLA_ERR_ARG, "out of host memory");
  const char* msg = "";
  int rc = mla::build_device_plan(batch, page_size, num_heads, q_len, num_sms, p, &msg);
  if (rc != MLA_OK) { delete p; return fail(rc, msg); }
  *plan_out = p;
  if (workspace_bytes_out) *workspace_bytes_out = p->ws_bytes;
  return ok();
}

int mla_plan_is_device(const mla_plan* plan) { return plan && plan->device ? 1 : 0; }

int mla_plan_read_device_schedule(const mla_plan* plan, const void* workspace, int32_t* out, int capacity,
                                  int* num_segments_out) {
  if (!plan || !plan->device || !workspace || !out || capacity < 0 || !num_segments_out)
    return fail(MLA_ERR_ARG, "bad arguments");
  mla::Schedule<mla::kSegCapLarge>* h = new (std::nothrow) mla::Schedule<mla::kSegCapLarge>();
  if (!h) return fail(MLA_ERR_ARG, "out of host memory");
  cudaError_t e = cudaMemcpy(h, static_cast<const char*>(workspace) + mla::kDevSchedOffset, sizeof(*h),
                             cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) {
    delete h;
    return fail(MLA_ERR_CUDA, std::string("reading the device schedule: ") + cudaGetErrorString(e));
  }
  const int n = std::max(0, std::min(h->num_segments, mla::kSegCapLarge));
  *num_segments_out = n;
  int w = 0, copied = 0;
  for (int i = 0; i < n && i < capacity; ++i) {
    while (w < h->num_workers && h->worker_seg[w + 1] <= i) ++w;
    out[5 * i + 0] = w;
    out[5 * i + 1] = h->seg[i].req;
    out[5 * i + 2] = h->seg[i].tile_begin;
    out[5 * i + 3] = h->seg[i].tile_end;
    out[5 * i + 4] = h->seg[i].slot;
    ++copied;
  }
  delete h;
  ok();
  return copied;
}

int mla_decode_fp8q(const mla_plan* plan, const void* q, int num_tokens, int num_heads, const void* kv_pages,
                    int64_t num_pages, int page_size, const int32_t* block_table, int bt_stride,
                    const int32_t* seq_lens, const int32_t* cu_seqlens_q, float scale, float k_scale, void* out,
                    float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  if (!q) return fail(MLA_ERR_ARG, "q is NULL");
  Prepared pr;
  // q stands in for both query pointers in the shared checks; the kernel
  // reads it as merged rows
  int rc = prepare(plan, q, q, num_tokens, num_heads, kv_pages, MLA_KV_E4M3, num_pages, page_size, block_table,
                   bt_stride, seq_lens, cu_seqlens_q, scale, k_scale, out, lse, workspace, workspace_bytes, &pr);
  if (rc != MLA_OK) return rc;
  if (!aligned(q, 16)) return fail(MLA_ERR_ARG, "q must be 16-byte aligned");
  pr.args.q_e4m3 = 1;
  pr.args.q_pe = nullptr;
  rc = check_device(nullptr);
  if (rc != MLA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  rc = launch_main(plan, pr, s);
  if (rc != MLA_OK) return rc;
  rc = launch_combine(plan, pr, s);
  return rc == MLA_OK ? ok() : rc;
}

size_t mla_plan_workspace_bytes(const mla_plan* plan) { return plan ? plan->ws_bytes : 0; }
int mla_plan_num_workers(const mla_plan* plan) { return plan ? plan->num_workers : 0; }
int mla_plan_num_segments(const mla_plan* plan) { return plan ? (int)plan->segs.size() : 0; }
int mla_plan_num_partial_slots(const mla_plan* plan) { return plan ? plan->num_slots : 0; }

int mla_plan_get_segments(const mla_plan* plan, int32_t* out, int capacity) {
  if (!plan || !out || capacity < 0) return fail(MLA_ERR_ARG, "bad arguments");
  const int n = std::min<int>(capacity, (int)plan->segs.size());
  for (int i = 0; i < n; ++i) {
    out[5 * i + 0] = plan->seg_worker[i];
    out[5 * i + 1] = plan->segs[i].req;
    out[5 * i + 2] = plan->segs[i].tile_begin;
    out[5 * i + 3] = plan->segs[i].tile_end;
    out[5 * i + 4] = plan->segs[i].slot;
  }
  return n;
}

void mla_planner_constants(int* tile_tokens, int* segment_overhead_tiles, int* min_split_tiles) {
  if (tile_tokens) *tile_tokens = mla::kTileTokens;
  if (segment_overhead_tiles) *segment_overhead_tiles = mla::kSegOverheadTiles;
  if (min_split_tiles) *min_split_tiles = mla::kMinSplitTiles;
}

const char* mla_decode_last_error_string(void) { return g_last_error.c_str(); }

int mla_decode_device_error(int* code, int reset) {
  if (!code) return fail(MLA_ERR_ARG, "code is NULL");
  int bt_code = 0, kw_code = 0;
  cudaError_t e = mla::sm103_read_error(code, reset != 0);
  if (e == cudaSuccess) e = mla::block_table_read_error(&bt_code, reset != 0);
  if (e == cudaSuccess) e = mla::kv_write_read_error(&kw_code, reset != 0);
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, std::string("reading the kernel error word: ") + cudaGetErrorString(e));
  if (*code == 0) *code = bt_code;
  if (*code == 0) *code = kw_code;
  return ok();
}

// Shared argument checks of the two block-table builders.
static int check_block_table_args(const int32_t* pool, int64_t pool_rows, int64_t pool_cols,
                                  const int32_t* req_pool_indices, int batch, int32_t* block_table,
                                  int max_blocks) {
  if (!pool || !req_pool_indices || !block_table) return fail(MLA_ERR_ARG, "a required device pointer is NULL");
  if (batch < 1 || batch > (1 << 24)) return fail(MLA_ERR_ARG, "batch must be in [1, 2^24]");
  if (max_blocks < 1 || max_blocks > MLA_BLOCK_TABLE_MAX_BLOCKS)
    return fail(MLA_ERR_ARG, "max_blocks must be in [1, MLA_BLOCK_TABLE_MAX_BLOCKS]");
  if (pool_rows < 1 || pool_cols < 1 || pool_rows > (INT64_MAX / pool_cols))
    return fail(MLA_ERR_ARG, "pool_rows and pool columns must be >= 1");
  if (!aligned(pool, 4) || !aligned(req_pool_indices, 4) || !aligned(block_table, 4))
    return fail(MLA_ERR_ARG, "int32 arrays must be 4-byte aligned");
  return check_device(nullptr);
}

int mla_block_table_from_tokens(const int32_t* req_to_token, int64_t pool_rows, int64_t token_cols,
                                const int32_t* req_pool_indices, const int32_t* seq_lens, int batch,
                                int page_size, int32_t* block_table, int max_blocks, void* stream) {
  if (page_size != 32 && page_size != 64) return fail(MLA_ERR_ARG, "page_size must be 32 or 64");
  if (!seq_lens || !aligned(seq_lens, 4)) return fail(MLA_ERR_ARG, "seq_lens must be a 4-byte aligned device pointer");
  int rc = check_block_table_args(req_to_token, pool_rows, token_cols, req_pool_indices, batch, block_table,
                                  max_blocks);
  if (rc != MLA_OK) return rc;
  cudaError_t e = mla::launch_block_table_from_tokens(req_to_token, pool_rows, token_cols, req_pool_indices,
                                                      seq_lens, batch, page_size, block_table, max_blocks,
                                                      static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, std::string("block-table launch: ") + cudaGetErrorString(e));
  return ok();
}

int mla_rope_quantize_cache_write(const void* q_nope, const void* q_rope, int num_tokens, int num_heads,
                                  void* q_out, int q_out_dtype, const void* k_nope, const void* k_rope,
                                  const int64_t* positions, const float* cos_sin_cache, int64_t max_position,
                                  int is_neox, void* kv_pages, int kv_dtype, int64_t num_pages, int page_size,
                                  const int64_t* out_cache_loc, void* stream) {
  if (num_tokens < 1 || num_heads < 0 || num_heads > (1 << 16)) return fail(MLA_ERR_ARG, "num_tokens >= 1, num_heads in [0, 65536]");
  // one flat grid of 256-thread blocks covers 72 items per (token, head or key) row
  if ((int64_t)num_tokens * (num_heads + 1) * 72 > (int64_t)INT32_MAX * 256)
    return fail(MLA_ERR_ARG, "too many tokens x heads for one launch");
  if (q_out_dtype != MLA_Q_BF16 && q_out_dtype != MLA_Q_E4M3) return fail(MLA_ERR_ARG, "q_out_dtype must be MLA_Q_BF16 or MLA_Q_E4M3");
  if (kv_dtype != MLA_KV_BF16 && kv_dtype != MLA_KV_E4M3) return fail(MLA_ERR_ARG, "kv_dtype must be MLA_KV_BF16 or MLA_KV_E4M3");
  if (page_size != 32 && page_size != 64) return fail(MLA_ERR_ARG, "page_size must be 32 or 64");
  if (num_pages <= 0 || num_pages * (int64_t)page_size > INT32_MAX) return fail(MLA_ERR_ARG, "num_pages must be > 0 and num_pages * page_size < 2^31");
  if (!k_nope || !k_rope || !kv_pages || !out_cache_loc) return fail(MLA_ERR_ARG, "a required device pointer is NULL");
  if (num_heads > 0 && (!q_rope || !q_out || (q_out_dtype == MLA_Q_E4M3 && !q_nope)))
    return fail(MLA_ERR_ARG, "query pointers are NULL");
  if (cos_sin_cache && (!positions || max_position < 1)) return fail(MLA_ERR_ARG, "positions / max_position missing");
  if (!aligned(k_nope, 16) || !aligned(k_rope, 16) || !aligned(kv_pages, 16) || !aligned(out_cache_loc, 8) ||
      (q_nope && !aligned(q_nope, 16)) || (q_rope && !aligned(q_rope, 16)) || (q_out && !aligned(q_out, 16)) ||
      (cos_sin_cache && !aligned(cos_sin_cache, 16)) || (positions && !aligned(positions, 8)))
    return fail(MLA_ERR_ARG, "arrays must be 16-byte aligned (index arrays 8-byte)");
  int rc = check_device(nullptr);
  if (rc != MLA_OK) return rc;
  cudaError_t e = mla::launch_rope_quantize_write(q_nope, q_rope, num_tokens, num_heads, q_out, q_out_dtype, k_nope,
                                                  k_rope, positions, cos_sin_cache, max_position, is_neox, kv_pages,
                                                  kv_dtype, num_pages, page_size, out_cache_loc,
                                                  static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, std::string("rope / cache-write launch: ") + cudaGetErrorString(e));
  return ok();
}

int mla_block_table_from_pages(const int32_t* req_to_page, int64_t pool_rows, int64_t page_cols,
                               const int32_t* req_pool_indices, int batch, int32_t* block_table,
                               int max_blocks, void* stream) {
  int rc = check_block_table_args(req_to_page, pool_rows, page_cols, req_pool_indices, batch, block_table,
                                  max_blocks);
  if (rc != MLA_OK) return rc;
  cudaError_t e = mla::launch_block_table_from_pages(req_to_page, pool_rows, page_cols, req_pool_indices, batch,
                                                     block_table, max_blocks, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, std::string("block-table launch: ") + cudaGetErrorString(e));
  return ok();
}

int mla_decode_version(void) { return 100; }

}  // extern "C"
