/*
 * mla_decode.h -- C ABI of the GB300 (sm_103a) paged MLA decode library.
 *
 * Operation.  Weight-absorbed Multi-head Latent Attention decode over a paged
 * latent KV cache, the call the serving pages make into their decode kernels
 * (sglang trtllm_mla_backend.py, TRTLLMMLABackend._run_decode_kernel /
 * forward_decode; tokenspeed trtllm_mla.py, forward_decode; tokenspeed
 * flashmla.py, FlashMLABackend.forward_decode and forward_extend).  For
 * request b with L = seq_lens[b] cache tokens, query position i < q_len and
 * head h (row t = b*q_len + i of the query):
 *
 *   visible keys   V = L - q_len + 1 + i          (bottom-right causal)
 *   cache row j    kv_pages[block_table[b][j / page_size]][j % page_size]
 *                  (576 wide: 512 latent c_kv, then 64 rotary k_pe)
 *   score          s_j = scale * kf * (q_nope[t,h,:] . c_kv_j + q_pe[t,h,:] . k_pe_j)
 *   out[t,h,:]     = kf * sum_{j<V} softmax(s)_j c_kv_j          (512 wide)
 *   lse[t,h]       = ln sum_{j<V} exp(s_j)                       (natural log)
 *
 * with kf = k_scale for an e4m3 cache and 1 for bf16 (tokenspeed
 * trtllm_mla.py, forward_decode: bmm1_scale = k_scale * layer.scaling; sglang
 * _compute_decode_bmm1_scale: k_scale applies to an FP8 cache only).  Rows
 * with V <= 0 give out = 0 and lse = -inf (sglang forward_extend: zero-KV rows
 * are forced to out=0, lse=-inf so a later merge ignores them).
 *
 * Work is split in two calls, as the pages plan (get_mla_metadata /
 * init_forward_metadata) before they run:
 *   1. mla_decode_plan   host, once per batch shape: split-KV schedule and
 *                        the workspace size it needs.
 *   2. mla_decode        device, asynchronous on the caller's stream: the
 *                        split-KV main kernel, then (if any request was split)
 *                        the LSE combine kernel.
 *
 * Conventions for every function below.
 *   - Return 0 on success or a negative MLA_ERR_* code; the message of the
 *     last failure on the calling thread is mla_decode_last_error_string().
 *   - Pointers marked "device" must be device memory of the current device;
 *     "host" pointers are ordinary host memory.  The caller owns every buffer.
 *   - Nothing in mla_decode allocates, frees or synchronises; all argument
 *     errors are detected on the host before any launch.
 *   - bf16 values are IEEE bfloat16, e4m3 values are OCP float8 e4m3fn.
 *
 * Precision.  Products run on the tensor cores with bf16 operands (fp16 for
 * an e4m3 cache, to which e4m3 and a bf16 query convert exactly) and fp32
 * accumulation.  Each score is the sum of two fp32 partial products, one of
 * which is rounded to 24 bits (relative error at most 2^-16) on its way
 * between the two CTAs that share the work.  Probabilities enter P.V as bf16
 * (fp16 for an e4m3 cache); the row sums and the lse use them unrounded.
 * Split requests merge bf16 partial outputs.  Against the exact float64
 * result the library is tested to max|out - ref| <= 1e-2 * max|ref| + 1e-3
 * and |lse - ref| <= 2e-3 (bf16 cache), and max|out - ref| <= 5e-2 * max|ref|
 * (e4m3 cache); rows with no visible key are exactly 0 and -inf.
 */
#ifndef MLA_DECODE_H_
#define MLA_DECODE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MLA_OK 0
#define MLA_ERR_ARG (-1)           /* bad argument (pointer, size, dtype, page size) */
#define MLA_ERR_WORKSPACE (-2)     /* workspace smaller than the plan needs */
#define MLA_ERR_PLAN_MISMATCH (-3) /* shapes differ from the ones planned for */
#define MLA_ERR_CUDA (-4)          /* a CUDA runtime call or launch failed */
#define MLA_ERR_UNSUPPORTED (-5)   /* device is not sm_103 or lacks a feature */

#define MLA_KV_BF16 0
#define MLA_KV_E4M3 1

#define MLA_KV_LORA_RANK 512
#define MLA_ROPE_DIM 64
#define MLA_KV_DIM 576

/* Opaque host object holding one split-KV schedule.  Created by
 * mla_decode_plan, released by mla_plan_destroy; read-only afterwards, so one
 * plan may serve concurrent mla_decode calls. */
typedef struct mla_plan mla_plan;

/*
 * Plan the split-KV schedule of one decode batch (the role of FlashMLA's
 * get_mla_metadata(seq_lens, num_heads * q_len, 1) in tokenspeed flashmla.py,
 * FlashMLABackend._init_decode_metadata: tile-scheduler metadata plus
 * num_splits[batch + 1]).
 *
 *   seq_lens_host  host int32[batch]: cache tokens per request, including the
 *                  q_len new tokens; 0 allowed.  Only read during the call.
 *   batch          >= 1 requests.
 *   page_size      32 or 64 tokens per cache page (the pages accept only
 *                  these: tokenspeed trtllm_mla.py, TRTLLMMLABackend.__init__).
 *   num_heads      query heads H >= 1; num_heads * q_len <= 128.
 *   q_len          query tokens per request, >= 1 (q_len > 1: speculative
 *                  verify / draft decode with the causal rule above).
 *   num_sms        SMs to schedule for; 0 = query the current device.
 *   plan_out       receives the new plan (caller frees with mla_plan_destroy).
 *   workspace_bytes_out  receives the device workspace size mla_decode needs
 *                  (0 when no request is split).
 *
 * The plan may also be made from upper bounds of the lengths: mla_decode
 * masks with the device seq_lens it is given, so a request that turns out
 * shorter only skips work (keys beyond the planned length are not visited).
 * Errors: MLA_ERR_ARG, MLA_ERR_CUDA (device query).
 */
int mla_decode_plan(const int32_t* seq_lens_host, int batch, int page_size, int num_heads,
                    int q_len, int num_sms, mla_plan** plan_out, size_t* workspace_bytes_out);

/* Release a plan (NULL is ignored). */
void mla_plan_destroy(mla_plan* plan);

/*
 * Run the decode on `stream` (a cudaStream_t; NULL = legacy default stream).
 *
 *   plan          from mla_decode_plan.
 *   q_nope        device bf16 [num_tokens, num_heads, 512], row-major; the
 *                 absorbed no-PE query (num_tokens = batch * q_len,
 *                 request-major then query position).
 *   q_pe          device bf16 [num_tokens, num_heads, 64], row-major.
 *   num_tokens, num_heads, page_size
 *                 must equal the plan's batch * q_len, num_heads and
 *                 page_size, else MLA_ERR_PLAN_MISMATCH (the pages re-plan
 *                 when the batch outgrew the plan: sglang forward_decode).
 *   kv_pages      device [num_pages, page_size, 576], row-major, element
 *                 type kv_dtype (MLA_KV_BF16 or MLA_KV_E4M3); 16-byte aligned.
 *   num_pages     pages in the pool (> 0).
 *   block_table   device int32 [batch, bt_stride], physical page ids; entries
 *                 past ceil(seq_len / page_size) are never read, so any
 *                 padding value (-1, 0, ...) is fine.  bt_stride must cover
 *                 the longest planned request.
 *   seq_lens      device int32 [batch]; lengths used for masking (see plan).
 *   scale         softmax scale, 1/sqrt(192) for DeepSeek-V3 shapes.
 *   k_scale       per-tensor dequantisation scale of an e4m3 cache (finite,
 *                 > 0); ignored for a bf16 cache, as the pages ignore a
 *                 checkpoint k_scale there (sglang _compute_decode_bmm1_scale).
 *   out           device bf16 [num_tokens, num_heads, 512]; fully written.
 *   lse           device fp32 [num_tokens, num_heads]; fully written.
 *   workspace     device scratch of >= the planned size, 256-byte aligned
 *                 (may be NULL when the planned size is 0).  No initial
 *                 contents are needed and none are kept between calls;
 *                 calls that overlap on the GPU must not share it.
 *
 * Errors: MLA_ERR_ARG, MLA_ERR_PLAN_MISMATCH, MLA_ERR_WORKSPACE,
 * MLA_ERR_UNSUPPORTED, MLA_ERR_CUDA (launch failure).  Kernel-side faults
 * surface as usual through the CUDA stream.
 */
int mla_decode(const mla_plan* plan, const void* q_nope, const void* q_pe, int num_tokens,
               int num_heads, const void* kv_pages, int kv_dtype, int64_t num_pages,
               int page_size, const int32_t* block_table, int bt_stride,
               const int32_t* seq_lens, float scale, float k_scale, void* out, float* lse,
               void* workspace, size_t workspace_bytes, void* stream);

/*
 * mla_decode for a caller whose per-step inputs and results live in host
 * memory (a serving loop that receives the new query on the host): on
 * `stream`, copy the step's inputs in, decode, and copy the results out.
 *
 *   q_nope_host, q_pe_host, block_table_host, seq_lens_host
 *                 host arrays shaped like q_nope, q_pe, block_table and
 *                 seq_lens of mla_decode; each is copied whole (one
 *                 cudaMemcpyAsync each) into the device buffer of the same
 *                 name, which this call therefore overwrites.
 *   out_host, lse_host
 *                 host arrays shaped like out and lse; the device results
 *                 are copied there after the decode.
 *   the rest      as for mla_decode (all device buffers).
 *
 * Returns once the work is queued: the host arrays must stay valid until the
 * stream has passed them, and the results are in out_host / lse_host only
 * after the caller synchronises with the stream (an event, say).  Pinned
 * host memory (cudaHostAlloc) lets the copies run asynchronously, so that
 * calls on two streams with two sets of buffers overlap one step's copies
 * with another step's decode; pageable memory works but the copies then
 * block the host.  Errors: those of mla_decode, MLA_ERR_ARG for a NULL host
 * pointer, MLA_ERR_CUDA when a copy cannot be queued.
 */
int mla_decode_host_io(const mla_plan* plan, void* q_nope, void* q_pe, int num_tokens, int num_heads,
                       const void* kv_pages, int kv_dtype, int64_t num_pages, int page_size,
                       int32_t* block_table, int bt_stride, int32_t* seq_lens, float scale, float k_scale,
                       void* out, float* lse, void* workspace, size_t workspace_bytes,
                       const void* q_nope_host, const void* q_pe_host, const int32_t* block_table_host,
                       const int32_t* seq_lens_host, void* out_host, float* lse_host, void* stream);

/*
 * The two launches of mla_decode, exposed separately so callers (and the
 * benchmark) can time or interleave them.  mla_decode == mla_decode_main
 * followed by mla_decode_combine on the same stream, with the same
 * arguments.  mla_decode_main writes the rows of unsplit requests to
 * out/lse and per-split partial results into the workspace;
 * mla_decode_combine merges the partials of split requests by their
 * log-sum-exp (lse = ln sum_k e^{lse_k}, out = sum_k e^{lse_k - lse} out_k;
 * splits with lse = -inf weigh nothing) and is a no-op without splits.
 */
int mla_decode_main(const mla_plan* plan, const void* q_nope, const void* q_pe, int num_tokens,
                    int num_heads, const void* kv_pages, int kv_dtype, int64_t num_pages,
                    int page_size, const int32_t* block_table, int bt_stride,
                    const int32_t* seq_lens, float scale, float k_scale, void* out, float* lse,
                    void* workspace, size_t workspace_bytes, void* stream);
int mla_decode_combine(const mla_plan* plan, void* out, float* lse, void* workspace,
                       size_t workspace_bytes, void* stream);

/*
 * Ragged query counts: a batch whose requests carry different numbers of
 * query tokens, packed back to back -- the draft-extend step after
 * speculative decoding, where each request keeps a different number of
 * accepted draft tokens (sglang trtllm_mla_backend.py, init_forward_metadata,
 * draft-extend branch: cu_seqlens_q = [0, cumsum(extend_seq_lens)]).
 *
 * Token i < q_b of request b (query row cu_seqlens_q[b] + i) sees
 *   V = L - q_b + 1 + i keys,  L = seq_lens[b],  q_b = cu_seqlens_q[b+1] - cu_seqlens_q[b],
 * the same bottom-right causal rule as mla_decode per request: exactly what
 * the pages obtain by padding every request's queries to the longest,
 * decoding with seq_lens_k = L - q_b + max_q and dropping the padding rows
 * (forward_extend, pad_draft_extend_query / unpad_draft_extend_output),
 * without the padding.
 *
 * mla_decode_plan_ragged: as mla_decode_plan with q_len = max(q_lens_host)
 * (at least 1; num_heads * that <= 128).  q_lens_host: host int32 [batch],
 * >= 0 (0 = a request with no query token); only read during the call.  The
 * device counts given to mla_decode_ragged may differ as long as none
 * exceeds that maximum.
 *
 * mla_decode_ragged: as mla_decode, except
 *   q_nope, q_pe, out, lse  hold num_tokens rows, 1 <= num_tokens <=
 *                 batch * max(q_lens); rows no request owns are not written.
 *   cu_seqlens_q  device int32 [batch + 1], nondecreasing, cu_seqlens_q[0] >= 0,
 *                 cu_seqlens_q[batch] <= num_tokens, each count <= the
 *                 planned maximum.  A request whose entry breaks this gets no
 *                 query row (nothing is read or written for it) and the error
 *                 word of mla_decode_device_error reads 0x501.
 * Errors: those of mla_decode; MLA_ERR_ARG also for a NULL cu_seqlens_q.
 * (mla_decode_main / mla_decode_combine are the uniform path only.)
 */
int mla_decode_plan_ragged(const int32_t* seq_lens_host, const int32_t* q_lens_host, int batch, int page_size,
                           int num_heads, int num_sms, mla_plan** plan_out, size_t* workspace_bytes_out);
int mla_decode_ragged(const mla_plan* plan, const void* q_nope, const void* q_pe, int num_tokens, int num_heads,
                      const void* kv_pages, int kv_dtype, int64_t num_pages, int page_size,
                      const int32_t* block_table, int bt_stride, const int32_t* seq_lens,
                      const int32_t* cu_seqlens_q, float scale, float k_scale, void* out, float* lse,
                      void* workspace, size_t workspace_bytes, void* stream);

/*
 * mla_decode_fp8q -- the decode of the pages' FP8 path: an e4m3 cache and
 * the merged e4m3 query that mla_rope_quantize_cache_write (MLA_Q_E4M3)
 * produces (sglang trtllm_mla_backend.py, forward_decode: the output of
 * mla_quantize_and_rope_for_fp8 goes to the decode kernel as
 * q.view(-1, H, 576); _compute_decode_bmm1_scale uses q_scale = 1).
 *
 *   q             device e4m3 [num_tokens, num_heads, 576] = [q_nope | q_pe],
 *                 16-byte aligned; no query scale.
 *   cu_seqlens_q  NULL for a uniform batch (num_tokens = batch * q_len), or
 *                 the ragged offsets of mla_decode_ragged.
 * Everything else as mla_decode with kv_dtype = MLA_KV_E4M3.  The query's
 * values are exact in fp16, so the result equals mla_decode's over the
 * same values given as bf16.
 */
int mla_decode_fp8q(const mla_plan* plan, const void* q, int num_tokens, int num_heads, const void* kv_pages,
                    int64_t num_pages, int page_size, const int32_t* block_table, int bt_stride,
                    const int32_t* seq_lens, const int32_t* cu_seqlens_q, float scale, float k_scale, void* out,
                    float* lse, void* workspace, size_t workspace_bytes, void* stream);

/*
 * mla_decode_noalloc -- the decode for callers that cannot allocate device
 * memory.  (No counterpart on the serving pages: their backends always own a
 * workspace buffer; this entry point is this library's own addition.)
 *
 * Same arguments and results as mla_decode, minus the workspace: the split
 * partials go to a scratch array built into the library (a fixed-size
 * __device__ variable of MLA_NOALLOC_SCRATCH_BYTES).  Meant for code that is
 * handed only its inputs and outputs and may not call cudaMalloc -- e.g. a
 * plugin running under a host framework's own memory manager, or an
 * allocation-free serving loop.  Nothing in this call allocates or frees.
 *
 *   - Plans needing more than MLA_NOALLOC_SCRATCH_BYTES of workspace are
 *     rejected with MLA_ERR_WORKSPACE (use mla_decode then).
 *   - The array is held by every device the code has been loaded on, until
 *     the process exits.
 *   - There is one array per device, shared by all calls on it; contents left
 *     by a previous call are never read before being rewritten, so nothing
 *     needs clearing, but calls that overlap on the GPU race: order them.
 *   - The array's device address is looked up (cudaGetSymbolAddress) the
 *     first time a call runs under a CUDA context, and cached under that
 *     context's unique id; a context made after cudaDeviceReset, or another
 *     context, looks it up again.  That first call may load the library's
 *     module in the context: make it before any stream capture.
 *   - Errors: those of mla_decode (MLA_ERR_UNSUPPORTED on a device that is
 *     not sm_103, checked before anything else); MLA_ERR_WORKSPACE for a
 *     plan larger than the array; MLA_ERR_CUDA if the address lookup fails.
 */
#define MLA_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
int mla_decode_noalloc(const mla_plan* plan, const void* q_nope, const void* q_pe, int num_tokens,
                       int num_heads, const void* kv_pages, int kv_dtype, int64_t num_pages,
                       int page_size, const int32_t* block_table, int bt_stride,
                       const int32_t* seq_lens, float scale, float k_scale, void* out, float* lse,
                       void* stream);

/*
 * Device plans: the split-KV schedule built on the device, from the device
 * seq_lens, at every decode.  A decode made with a device plan can be
 * captured in a CUDA graph once per batch shape and replayed for any
 * lengths: there is no host copy of the lengths and nothing to re-plan
 * (what FlashMLA's get_mla_metadata does on the device for tokenspeed
 * flashmla.py, _init_decode_metadata; padded graph rows keep the pages'
 * seq_len fill value of 1, P1 get_cuda_graph_seq_len_fill_value, and cost
 * one tile).
 *
 * mla_decode_plan_device: the batch shape only (batch 1 .. 1793, page_size,
 *   num_heads, q_len -- the maximum count for mla_decode_ragged -- and
 *   num_sms as in mla_decode_plan).  The workspace it asks for holds the
 *   schedule and the partials of the largest schedule any lengths can give
 *   (2 (W - 1) split slots for W = num_sms / 2 workers).
 * mla_decode, mla_decode_ragged, mla_decode_noalloc, mla_decode_main and
 *   mla_decode_combine accept it: mla_decode_main (and so mla_decode) first
 *   launches the planner kernel on the stream, which writes the schedule
 *   into the workspace head; the main kernel reads it there.  Any bt_stride
 *   >= 1 is accepted; lengths are clamped to bt_stride * page_size keys.
 *   The schedule follows a fixed rule (mla_plan_device.cu): the same lengths
 *   always give the same schedule, and so bit-identical results.
 * mla_plan_is_device: 1 for a device plan, else 0.
 * mla_plan_read_device_schedule: copy the schedule the last decode built in
 *   `workspace` to host int32 out[5 * capacity], as mla_plan_get_segments
 *   does; *num_segments_out receives its length.  Synchronous (a blocking
 *   device-to-host copy): for tests and inspection.  Returns the number
 *   copied or a negative MLA_ERR_* code.
 * The host-plan inspection calls (mla_plan_num_segments,
 * mla_plan_get_segments) report 0 segments for a device plan, and
 * mla_plan_num_partial_slots its 2 (W - 1) slot capacity.
 */
int mla_decode_plan_device(int batch, int page_size, int num_heads, int q_len, int num_sms, mla_plan** plan_out,
                           size_t* workspace_bytes_out);
int mla_plan_is_device(const mla_plan* plan);
int mla_plan_read_device_schedule(const mla_plan* plan, const void* workspace, int32_t* out, int capacity,
                                  int* num_segments_out);

/* ---- RoPE + FP8 quantisation + paged cache write (the step before) ----
 *
 * One launch, asynchronous on `stream`, for the new tokens of a decode step:
 * rotary embedding of the rope parts of the query and of the key, the query
 * output, and each token's key row written into its cache slot.  The pages'
 * FP8 path does this with mla_quantize_and_rope_for_fp8 followed by
 * set_mla_kv_buffer (sglang trtllm_mla_backend.py, forward_decode; tokenspeed
 * trtllm_mla.py, forward_decode stores k[..., :512] and k[..., 512:]).
 *
 *   q_nope        device bf16 [num_tokens, num_heads, 512] (read only for
 *                 MLA_Q_E4M3).
 *   q_rope        device bf16 [num_tokens, num_heads, 64].
 *   num_heads     query heads; 0 = no query work (a plain cache write).
 *   q_out         MLA_Q_E4M3: device e4m3 [num_tokens, num_heads, 576] =
 *                 [q_nope | rope(q_rope)], the merged FP8 query of the pages;
 *                 MLA_Q_BF16: device bf16 [num_tokens, num_heads, 64] =
 *                 rope(q_rope), the q_pe that mla_decode takes beside q_nope.
 *   k_nope, k_rope  device bf16 [num_tokens, 512] and [num_tokens, 64].
 *   positions     device int64 [num_tokens] rows of cos_sin_cache (may be
 *                 NULL when cos_sin_cache is NULL).
 *   cos_sin_cache device fp32 [max_position, 64]: 32 cosines then 32 sines
 *                 per position, 16-byte aligned; NULL = no rotation.
 *   is_neox       nonzero: element i pairs with i + 32; zero: 2i with 2i + 1.
 *                 A pair (a, b) becomes (a cos - b sin, b cos + a sin), in
 *                 fp32 with every product and sum rounded on its own.
 *   kv_pages, kv_dtype, num_pages, page_size  the cache as mla_decode takes
 *                 it; token t's row [k_nope | rope(k_rope)] is written at
 *                 slot out_cache_loc[t] (device int64 [num_tokens]): row
 *                 slot % page_size of page slot / page_size.  Slots must be
 *                 distinct (two tokens writing one slot race, as any scatter).
 * FP8 values are rounded to nearest (ties to even) and saturate at +-448,
 * with no scale (the pages pass none); bf16 values round to nearest even.
 * Device-side errors (mla_decode_device_error): a position outside
 * [0, max_position) leaves that token's outputs unwritten (0x601); a slot
 * outside the cache leaves its key row unwritten (0x602).  Host-side:
 * MLA_ERR_ARG (also when num_tokens * (num_heads + 1) * 72 exceeds the
 * (2^31 - 1) * 256 items one launch covers), MLA_ERR_UNSUPPORTED,
 * MLA_ERR_CUDA.
 */
#define MLA_Q_BF16 0
#define MLA_Q_E4M3 1
int mla_rope_quantize_cache_write(const void* q_nope, const void* q_rope, int num_tokens, int num_heads,
                                  void* q_out, int q_out_dtype, const void* k_nope, const void* k_rope,
                                  const int64_t* positions, const float* cos_sin_cache, int64_t max_position,
                                  int is_neox, void* kv_pages, int kv_dtype, int64_t num_pages, int page_size,
                                  const int64_t* out_cache_loc, void* stream);

/* ---- block-table construction (the step before the decode) ----
 *
 * Build the [batch, max_blocks] int32 block table mla_decode reads from a
 * serving-side request pool, on the device and asynchronously on `stream`
 * (no host synchronisation, so both may be captured in a CUDA graph with the
 * decode).  The serving pages do this right before the decode: sglang
 * trtllm_mla_backend.py, TRTLLMMLABackend._create_block_kv_indices (a token
 * pool, create_flashmla_kv_indices_triton) and tokenspeed trtllm_mla.py,
 * TRTLLMMLABackend._create_block_kv_indices / tokenspeed flashmla.py,
 * _init_decode_metadata (a page pool, req_to_page[req_pool_indices]).
 *
 * Shared arguments:
 *   req_pool_indices  device int32 [batch]: pool row of each request.
 *   batch             requests, 1 .. 2^24.
 *   block_table       device int32 [batch, max_blocks], row-major; every
 *                     entry is written.
 *   max_blocks        1 .. MLA_BLOCK_TABLE_MAX_BLOCKS.
 * All int32 arrays 4-byte aligned; the caller owns every buffer.
 *
 * Device-side errors.  A pool row index outside [0, pool_rows), a lookup past
 * the pool's columns, a negative length or a negative token slot is not
 * read: the entry gets the padding value and the first such event since the
 * last reset is recorded in the word mla_decode_device_error reports
 * (0x301 row index, 0x302 column, 0x303 negative seq_len, 0x304 negative
 * slot).  Host-side errors: MLA_ERR_ARG, MLA_ERR_UNSUPPORTED, MLA_ERR_CUDA.
 */
#define MLA_BLOCK_TABLE_MAX_BLOCKS (65535 * 256)

/*
 * From a token pool: req_to_token is device int32 [pool_rows, token_cols],
 * row-major, the cache slot of each token of a pool row, where slot =
 * page_id * page_size + offset in the page (the cache viewed as
 * [num_pages, page_size, 576]).  With L = seq_lens[b] (device int32
 * [batch]):
 *   block_table[b][i] = req_to_token[req_pool_indices[b]][i * page_size] / page_size
 *                                              for i < ceil(L / page_size),
 *                     = -1                     otherwise
 * (the page of the first token of each of the request's pages).
 * page_size: 32 or 64.
 */
int mla_block_table_from_tokens(const int32_t* req_to_token, int64_t pool_rows, int64_t token_cols,
                                const int32_t* req_pool_indices, const int32_t* seq_lens, int batch,
                                int page_size, int32_t* block_table, int max_blocks, void* stream);

/*
 * From a page pool: req_to_page is device int32 [pool_rows, page_cols],
 * row-major, the page ids of each pool row.
 *   block_table[b][i] = req_to_page[req_pool_indices[b]][i]   for i < min(max_blocks, page_cols),
 *                     = 0                                     otherwise.
 */
int mla_block_table_from_pages(const int32_t* req_to_page, int64_t pool_rows, int64_t page_cols,
                               const int32_t* req_pool_indices, int batch, int32_t* block_table,
                               int max_blocks, void* stream);

/* ---- plan inspection (host only; used by tests and tools) ---- */

/* Device workspace bytes the plan needs. */
size_t mla_plan_workspace_bytes(const mla_plan* plan);
/* Workers (persistent CTA pairs) the plan schedules for. */
int mla_plan_num_workers(const mla_plan* plan);
/* Number of segments (work items).  A segment is one contiguous run of
 * 64-token tiles of one request, processed by one worker. */
int mla_plan_num_segments(const mla_plan* plan);
/* Copy the segments into host int32 out[5 * capacity] as
 * (worker, request, tile_begin, tile_end, partial_slot) tuples in execution
 * order; partial_slot = -1 when the request has a single segment and is
 * written directly.  Returns the number copied or MLA_ERR_ARG. */
int mla_plan_get_segments(const mla_plan* plan, int32_t* out, int capacity);
/* Number of partial-result slots in the workspace (sum of the split counts
 * of split requests). */
int mla_plan_num_partial_slots(const mla_plan* plan);

/* Planner constants: tokens per tile, per-segment overhead charged in tiles,
 * shortest piece a split request is cut into (in tiles). */
void mla_planner_constants(int* tile_tokens, int* segment_overhead_tiles, int* min_split_tiles);

/* Kernel-side error word of the current device: 0, or the code of the first
 * bounded wait that timed out inside a decode kernel since the last reset
 * (the kernel then stopped early and its outputs are not valid); failing
 * that, the first out-of-range lookup of a block-table builder (0x30x) or of
 * the RoPE / cache-write step (0x60x).  Reading it
 * synchronises with the device; reset != 0 clears it.  Errors: MLA_ERR_ARG,
 * MLA_ERR_CUDA. */
int mla_decode_device_error(int* code, int reset);

/* Message of the last failure on the calling thread ("" if none). */
const char* mla_decode_last_error_string(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int mla_decode_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_H_ */
