/*
 * bsxattn.h - C ABI of the XAttention block-sparse chunked-prefill library
 * for GB300 (sm_103a).
 *
 * The library implements one chunk of XAttention chunked prefill as described
 * by the nano-vllm pages (docs/xattention_algorithm_guide.md, "算法流程";
 * nanovllm/kvcache/sparse/xattn_bsa.py, XAttentionBSAPolicy.select_blocks and
 * compute_chunked_prefill):
 *
 *   bsx_xattn_estimate       stride-S antidiagonal scores, causal row softmax,
 *                            128-token block sums and threshold selection
 *                            -> uint8 block mask
 *   bsx_bsa_prefill          causal GQA block-sparse attention over the
 *                            selected 128-token blocks -> O and LSE
 *   bsx_merge_attn           LSE merge of two partial (O, LSE) pairs
 *   bsx_map_mask_to_cpu_blocks  1024-token CPU-block keep flags
 *   bsx_chunk_step           the whole chunk step on device inputs (the four
 *                            steps; one kernel launch where supported)
 *   bsx_chunk_prefill        estimate + attention over every key block (the
 *                            merge identity; one kernel launch where supported)
 *   bsx_chunk_step_host      the whole chunk step from host inputs to host
 *                            outputs (uploads, the four steps, read-back)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Tensors are caller-owned, contiguous, device-resident (CUDA global
 *    memory) and 16-byte aligned; bsx_chunk_step_host alone also takes host
 *    buffers and copies to and from them.  The library never allocates
 *    device memory or frees it, and never synchronises: work is enqueued on
 *    `stream` (a cudaStream_t; NULL means the legacy default stream) and the
 *    call returns.
 *  - Layouts are token-major:
 *        q     [B, q_len, Hq, d]            element type `dtype`
 *        k, v  [B, Lk, Hkv, d]              Lk = q_start_pos + q_len
 *        mask  [B, Hq, q_len/128, Lk/128]   uint8, 1 = block selected
 *        o     [B, q_len, Hq, d]            element type `dtype`
 *        lse   [B, Hq, q_len]               float32, natural log
 *    GQA: q-head h reads kv-head h / (Hq/Hkv).
 *  - q_start_pos is the absolute position of the chunk's first query; keys
 *    are all earlier tokens plus the chunk.  q_start_pos and q_len must be
 *    multiples of 128 (the BSA block size, fixed at 128 on the pages).
 *  - Arguments are validated on the host before any launch; a bad argument
 *    returns BSX_ERR_INVALID_ARG and an unsupported combination (dtype, d,
 *    stride; Lk above 2^24; a block mask of more than 2^31 - 1 elements,
 *    B * Hq * (q_len/128) * (Lk/128), for the calls that use one) returns
 *    BSX_ERR_UNSUPPORTED, with nothing enqueued.  There is no
 *    fallback path.  A CUDA launch error returns BSX_ERR_CUDA.  Errors the
 *    kernels detect asynchronously (a bounded wait that expired) are
 *    recorded in a device error word read by bsx_last_error().
 */
#ifndef BSXATTN_H_
#define BSXATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  BSX_OK = 0,
  BSX_ERR_INVALID_ARG = -1,
  BSX_ERR_UNSUPPORTED = -2,
  BSX_ERR_CUDA = -3,
  BSX_ERR_TIMEOUT = -4,
  BSX_ERR_WORKSPACE = -5
} bsx_status;

/*
 * Element types.  BSX_F8E4M3 (fp8: 1 sign, 4 exponent, 3 mantissa bits, no
 * infinities, largest finite value 448) is accepted by bsx_xattn_estimate and
 * bsx_xattn_estimate_noalloc only, for q and k with d = 128: the estimator's
 * reduced-precision operands (the pages keep the estimator in the model
 * dtype; e4m3 K halves its largest input).  bsx_quantize_e4m3 makes them.
 */
typedef enum { BSX_F32 = 0, BSX_BF16 = 1, BSX_F8E4M3 = 2 } bsx_dtype;

/* Problem shape shared by all calls.  Hq % Hkv == 0; d in {64, 128}. */
typedef struct {
  int B;      /* batch (sequences of equal length and equal q_start_pos) */
  int Hq;     /* query heads */
  int Hkv;    /* key/value heads */
  int d;      /* head dimension */
  int dtype;  /* bsx_dtype of q, k, v and o */
} bsx_shape;

/* Flags for bsx_map_mask_to_cpu_blocks. */
#define BSX_FORCE_FIRST_LAST 1

/* Library version, (major << 16) | minor. */
int bsx_version(void);

/* Static description of a status code.  Never NULL. */
const char* bsx_status_string(int status);

/*
 * Bytes of device scratch bsx_xattn_estimate needs for this problem: one
 * float per (batch, q-head, key block, reshaped query row), i.e.
 * B * Hq * (Lk/128) * (q_len/stride) * 4.  Returns 0 for invalid arguments.
 */
size_t bsx_estimate_workspace_bytes(bsx_shape s, int q_len, int q_start_pos,
                                    int stride);

/*
 * XAttention estimate + block selection for one Q chunk.
 *
 * Defined by docs/xattention_algorithm_guide.md "算法流程" Phases 1-3 and
 * "块选择算法 (find_blocks_chunked)", with the chunk offset of xattn_bsa.py
 * select_blocks Steps 0-4:
 *   reshaped row I = q_start_pos/S + i (i < q_len/S), reshaped key J < Lk/S;
 *   s[I,J] = sum_{t<S} q[I*S+S-1-t] . k[J*S+t]                 (inverse mode)
 *   p[I,:] = softmax over J <= I of s[I,J] / (sqrt(d) * S)
 *   A[qb,kb] = sum of p over the (128/S) rows of q-block qb and the
 *              (128/S) columns of key block kb
 *   per (b, h, qb): blocks 0 and diag = q_start_pos/128 + qb are kept; the
 *   others are taken by descending A (ties: lower kb first) while the
 *   cumulative mass (forced blocks included) is below threshold * sum(A);
 *   the block that crosses the threshold is kept; threshold >= 1 keeps every
 *   causal block; blocks after the diagonal are never kept.
 *
 * q [B,q_len,Hq,d], k [B,Lk,Hkv,d] (device, `s.dtype`: f32, bf16, or e4m3
 * bytes with d = 128; with e4m3 the scores are those of the e4m3 values,
 * accumulated in fp32).
 * mask (out, device) uint8 [B, Hq, q_len/128, Lk/128]; every byte written.
 * block_sums (out, device, nullable) float32 [B, Hq, q_len/128, Lk/128]:
 *   A for kb <= diag, 0 after it.
 * workspace (device) of at least bsx_estimate_workspace_bytes() bytes,
 *   overwritten; else BSX_ERR_WORKSPACE.
 * stride in {4, 8, 16}; 0 < threshold.
 */
int bsx_xattn_estimate(bsx_shape s, const void* q, const void* k, int q_len,
                       int q_start_pos, int stride, float threshold,
                       uint8_t* mask, float* block_sums, void* workspace,
                       size_t workspace_bytes, void* stream);

/*
 * bf16 -> e4m3: dst[i] = the e4m3 value nearest to src[i] (ties to even
 * mantissa), values beyond +-448 saturated to +-448, for i < n.
 * src (device) bf16 [n]; dst (out, device) uint8 [n] (e4m3 bit patterns).
 * Enqueued on `stream`; n == 0 enqueues nothing; NULL pointers with n > 0 or
 * n < 0 are BSX_ERR_INVALID_ARG.  Any alignment (16-byte aligned src and
 * 8-byte aligned dst with n % 8 == 0 take the faster path).
 */
int bsx_quantize_e4m3(const void* src, uint8_t* dst, long long n, void* stream);

/*
 * bsx_xattn_estimate without a caller-provided workspace.  The pages have no
 * counterpart to this call; it exists for callers that may not allocate
 * device memory (a host engine that owns all device memory through its own
 * pool and forbids its plugins to call cudaMalloc, or a loop that may not
 * call an allocator) and have no buffer to lend as scratch.
 *
 * Same arguments, outputs and results as bsx_xattn_estimate, minus
 * `workspace`/`workspace_bytes`.  The scratch is a fixed 32 MiB array in
 * the library's own device code, held in global memory of every device that
 * uses it until the process exits.  A problem whose
 * bsx_estimate_workspace_bytes() exceeds 32 MiB (33554432 bytes) returns
 * BSX_ERR_WORKSPACE with nothing enqueued.
 * The first call on a device (with that device current) looks up the
 * array's device address and caches it.  CUDA loads the library's device
 * code lazily, so that first call is also when the 32 MiB are committed on
 * the device: it can fail for lack of device memory (BSX_ERR_CUDA, the CUDA
 * error printed to stderr).  Make it before the host engine fills its memory
 * pool, and before any stream capture.  The cached address belongs to the
 * device's primary context: after cudaDeviceReset, or from another driver
 * context, it is stale and must not be used.  All calls share the array:
 * calls whose work overlaps on the GPU (other streams, other host threads)
 * race on it and must be serialised by the caller.  Nothing in it needs to
 * start at zero (every cell read is first written by the same call).  This
 * call allocates nothing.
 */
int bsx_xattn_estimate_noalloc(bsx_shape s, const void* q, const void* k,
                               int q_len, int q_start_pos, int stride,
                               float threshold, uint8_t* mask,
                               float* block_sums, void* stream);

/*
 * Block-sparse causal attention (BSA) over key blocks [kb_begin, kb_end).
 *
 * Defined by docs/xattention_algorithm_guide.md "BSA (Block Sparse
 * Attention)" (block_sparse_attn_func with is_causal, 128-token blocks,
 * per-head block mask) and xattn_bsa.py compute_chunked_prefill (history and
 * current chunk computed separately, each returning O and LSE):
 *   query row i (position q_start_pos + i) of head h sees key j iff
 *   kb_begin*128 <= j < kb_end*128, j <= q_start_pos + i and
 *   mask[b, h, i/128, j/128] != 0;
 *   o[b,i,h,:] = sum_j softmax_j(q.k_j / sqrt(d)) v_j,
 *   lse[b,h,i] = ln sum_j exp(q.k_j / sqrt(d)).
 * A row that sees no key gets o = 0 and lse = -inf.
 * 0 <= kb_begin <= kb_end <= Lk/128 (an empty range is allowed).
 * o (out) [B,q_len,Hq,d] in `s.dtype`; lse (out) float32 [B,Hq,q_len].
 */
int bsx_bsa_prefill(bsx_shape s, const void* q, const void* k, const void* v,
                    const uint8_t* mask, int q_len, int q_start_pos,
                    int kb_begin, int kb_end, void* o, float* lse,
                    void* stream);

/*
 * Both parts of one chunk's block-sparse attention in a single launch: the
 * history, key blocks [0, q_start_pos/128), into (o_hist, lse_hist), and the
 * current chunk, key blocks [q_start_pos/128, Lk/128), into (o_curr,
 * lse_curr).  Each part is exactly what bsx_bsa_prefill computes for that
 * range (xattn_bsa.py compute_chunked_prefill attends to the history and to
 * the current chunk separately and merges the two by LSE, bsx_merge_attn).
 * One launch lets the short current-chunk work fill the tail of the history
 * work on the GPU.  Arguments, layouts and errors as bsx_bsa_prefill; the
 * four outputs must not overlap.  With q_start_pos == 0 the history part is
 * empty (o_hist = 0, lse_hist = -inf).
 */
int bsx_bsa_prefill_split(bsx_shape s, const void* q, const void* k, const void* v,
                          const uint8_t* mask, int q_len, int q_start_pos,
                          void* o_hist, float* lse_hist, void* o_curr, float* lse_curr,
                          void* stream);

/*
 * Bytes of device workspace bsx_chunk_prefill and bsx_chunk_step need: the
 * estimate partials of bsx_estimate_workspace_bytes(), rounded up to 256
 * bytes; then a control block of 4 * (4 + B * Hq * (ceil(R / 128) +
 * q_len / 128)) bytes rounded up to 256 (the fused launch's counters and
 * ready flags), with R = q_len / stride; then 4 * B * Hq * n_kt * R bytes rounded up to 256, n_kt =
 * (q_start_pos / stride + R - 1) / 256 + 1 (each reshaped row's
 * log-sum-exp over each 256-key tile, which the fused selection reads).
 * Returns 0 for invalid arguments.
 */
size_t bsx_chunk_prefill_workspace_bytes(bsx_shape s, int q_len, int q_start_pos,
                                         int stride);

/*
 * One chunk of XAttention prefill with the KV resident on the device:
 * bsx_xattn_estimate followed by bsx_bsa_prefill over every key block
 * [0, Lk/128).  By the merge identity this equals attending to the history
 * and the current chunk separately and merging them by LSE (the structure of
 * xattn_bsa.py compute_chunked_prefill), without the merge.
 *
 * docs/xattention_algorithm_guide.md "算法流程": estimate, select, attend, in
 * that order, for one chunk.  In bf16 with at most 1024 key blocks (Lk <=
 * 131072) the three stages run as ONE kernel launch (preceded by a 4-byte-
 * granular memset of the control block on the same stream): CTAs take
 * roles in the order they start -- estimate workers, which also select each
 * row once its estimate tiles are complete, then one attention CTA per
 * 128-row query tile, which waits for its row's mask; every such wait is
 * bounded (a wait that gives up sets the device error word, kernel id 3, and
 * ends the other waits; bsx_last_error).  Otherwise (f32, or more key blocks)
 * the estimate and the attention are separate launches.  The mask, o and lse
 * are those of the separate calls (the fused selection adds its row sums in
 * another order, which can only change near-threshold rows).
 *
 * Outputs: mask (as bsx_xattn_estimate), o, lse (as bsx_bsa_prefill).
 * Arguments are validated before anything is enqueued.  workspace (device,
 * 16-byte aligned) of at least bsx_chunk_prefill_workspace_bytes() bytes,
 * overwritten; else BSX_ERR_WORKSPACE.  Calls that overlap on the GPU need
 * separate workspaces.
 */
int bsx_chunk_prefill(bsx_shape s, const void* q, const void* k, const void* v,
                      int q_len, int q_start_pos, int stride, float threshold,
                      uint8_t* mask, void* o, float* lse, void* workspace,
                      size_t workspace_bytes, void* stream);

/*
 * One chunk step of XAttention chunked prefill with the KV resident on the
 * device, as the pages structure it (xattn_bsa.py compute_chunked_prefill and
 * select_blocks): bsx_xattn_estimate; bsx_bsa_prefill_split with the history
 * into (o, lse) and the current chunk into (o_curr, lse_curr);
 * bsx_merge_attn of the two into (o, lse); and, when keep is not NULL and
 * q_start_pos >= cpu_block_tokens, bsx_map_mask_to_cpu_blocks into keep (no
 * first/last forcing).
 *
 * In bf16 with at most 1024 key blocks (Lk <= 131072) the whole step is ONE
 * kernel launch (after memsets of its control block and of keep on the same
 * stream): the fused launch of bsx_chunk_prefill, whose attention CTA for a
 * query tile attends to the history and to the current chunk as two ranges
 * and merges the two results itself, and whose selection writes the keep
 * flags.  Otherwise the steps run as the separate launches listed above.
 * Results: the merged (o, lse) and keep bit for bit as the separate calls
 * give them on the kernel's mask; the mask as bsx_chunk_prefill's (the fused
 * selection adds its row sums in another order than bsx_xattn_estimate,
 * which can only change near-threshold rows); o_curr / lse_curr are
 * scratch, with unspecified contents afterwards.  With q_start_pos == 0 there is no
 * history and (o, lse) are the current chunk's.
 *
 * Arguments are validated before anything is enqueued; every buffer 16-byte
 * aligned; cpu_block_tokens (used only with keep) a positive multiple of 128
 * dividing q_start_pos.  workspace of at least
 * bsx_chunk_prefill_workspace_bytes() bytes, else BSX_ERR_WORKSPACE.
 */
int bsx_chunk_step(bsx_shape s, const void* q, const void* k, const void* v, int q_len,
                   int q_start_pos, int stride, float threshold, int cpu_block_tokens,
                   uint8_t* mask, void* o, float* lse, void* o_curr, float* lse_curr,
                   uint8_t* keep, void* workspace, size_t workspace_bytes, void* stream);

/*
 * LSE merge of two partial attentions over disjoint key sets, in place into
 * (o1, lse1).
 *
 * Defined by the nano-vllm optimization guide, "Online Softmax Merge -
 * Triton Fused Kernel" (merge_attention_outputs):
 *   m = max(lse1, lse2); w_i = exp(lse_i - m);
 *   o1 <- (w1*o1 + w2*o2) / (w1 + w2); lse1 <- m + ln(w1 + w2).
 * Rows whose two LSEs are both -inf get o1 = 0, lse1 = -inf.
 * o1 (in/out), o2 (in) [B,q_len,Hq,d] in `s.dtype`; lse1 (in/out), lse2 (in)
 * float32 [B,Hq,q_len].  o2/lse2 must not overlap o1/lse1.
 */
int bsx_merge_attn(bsx_shape s, int q_len, void* o1, float* lse1,
                   const void* o2, const float* lse2, void* stream);

/*
 * CPU-block keep flags from a BSA block mask.
 *
 * Defined by nano-vllm task_plan.md "核心设计理解" section 1 (a 1024-token
 * CPU block holds 8 BSA blocks) and section 3 (a CPU block is kept if any of
 * its BSA blocks is selected, OR over heads and q-blocks), and xattn_bsa.py
 * select_blocks Step 6 (history blocks only; first and last always added):
 *   keep[b,c] = OR_{h, qb, u < cpu_block_tokens/128}
 *               mask[b, h, qb, c*cpu_block_tokens/128 + u],
 *   for the history blocks c < q_start_pos / cpu_block_tokens.
 * flags & BSX_FORCE_FIRST_LAST also sets the first and last history block.
 * cpu_block_tokens: a positive multiple of 128 dividing q_start_pos.
 * keep (out, device) uint8 [B, q_start_pos / cpu_block_tokens].
 */
int bsx_map_mask_to_cpu_blocks(bsx_shape s, const uint8_t* mask, int q_len,
                               int q_start_pos, int cpu_block_tokens,
                               int flags, uint8_t* keep, void* stream);

/*
 * Block mask of the pages' CPU-offload attention, from CPU-block keep flags.
 *
 * nano-vllm xattn_bsa.py compute_chunked_prefill attends, for every head and
 * query, densely to all keys of the selected CPU blocks of the history (each
 * through flash_attn_with_lse without causal masking, merged by LSE) and
 * causally to the current chunk; select_blocks Step 6 picks the CPU blocks
 * (bsx_map_mask_to_cpu_blocks with BSX_FORCE_FIRST_LAST).  This call writes
 * the BSA block mask that makes bsx_bsa_prefill compute exactly that:
 *   mask[b,h,qb,kb] = keep[b, kb*128 / cpu_block_tokens]   kb < q_start_pos/128
 *                   = (kb <= q_start_pos/128 + qb)          otherwise.
 * keep (in, device) uint8 [B, q_start_pos / cpu_block_tokens] (may be NULL
 * when q_start_pos is 0); mask (out, device) uint8 [B, Hq, q_len/128,
 * Lk/128], every byte written.
 */
int bsx_cpu_block_mask(bsx_shape s, const uint8_t* keep, int q_len,
                       int q_start_pos, int cpu_block_tokens, uint8_t* mask,
                       void* stream);

/* Flags for bsx_chunk_step_host (BSX_FORCE_FIRST_LAST applies there too). */
#define BSX_STEP_OFFLOAD 2        /* attention of the pages' CPU-offload mode */
#define BSX_STEP_E4M3_ESTIMATE 4  /* estimator on e4m3 copies of q and k */
#define BSX_STEP_FUSED 8          /* one attention launch over all key blocks */

/* Caller-owned device buffers of bsx_chunk_step_host (16-byte aligned). */
typedef struct {
  void* q;                /* [B,q_len,Hq,d]  receives q_host */
  void* k;                /* [B,Lk,Hkv,d]    receives k_host */
  void* v;                /* [B,Lk,Hkv,d]    receives v_host */
  uint8_t* mask;          /* [B,Hq,q_len/128,Lk/128]  the estimator's mask */
  uint8_t* bsa_mask;      /* same shape; BSX_STEP_OFFLOAD only, else NULL */
  void* o;                /* [B,q_len,Hq,d]  history part, then the merged O */
  float* lse;             /* [B,Hq,q_len]    history part, then the merged LSE */
  void* o_curr;           /* [B,q_len,Hq,d]  current-chunk part; unused if fused */
  float* lse_curr;        /* [B,Hq,q_len]    current-chunk part; unused if fused */
  uint8_t* keep;          /* [B,q_start_pos/cpu_block_tokens] or NULL (no flags) */
  uint8_t* q8;            /* [B,q_len,Hq,d] e4m3; BSX_STEP_E4M3_ESTIMATE only */
  uint8_t* k8;            /* [B,Lk,Hkv,d]   e4m3; BSX_STEP_E4M3_ESTIMATE only */
  void* workspace;        /* bsx_estimate_workspace_bytes(s, ...) bytes, or
                             bsx_chunk_prefill_workspace_bytes() for a step
                             that runs as bsx_chunk_prefill (BSX_STEP_FUSED) */
  size_t workspace_bytes;
  void* done;             /* a cudaEvent_t, or NULL; see bsx_chunk_step_host */
} bsx_chunk_buffers;

/*
 * One chunk step of XAttention chunked prefill from host memory to host
 * memory: the structure of nano-vllm xattn_bsa.py (select_blocks, then
 * compute_chunked_prefill) with every input uploaded and every result read
 * back inside the call's stream work.
 *
 *   q_host [B,q_len,Hq,d], k_host / v_host [B,Lk,Hkv,d]  (in, host, `s.dtype`)
 *   -> upload into dev->q, dev->k, dev->v
 *   -> bsx_xattn_estimate -> dev->mask
 *   -> bsx_bsa_prefill_split -> (dev->o, dev->lse), (dev->o_curr, dev->lse_curr)
 *   -> bsx_merge_attn into (dev->o, dev->lse)
 *   -> bsx_map_mask_to_cpu_blocks -> dev->keep   (when dev->keep is not
 *      NULL and q_start_pos >= cpu_block_tokens)
 *   -> o_host [B,q_len,Hq,d], lse_host [B,Hq,q_len] float32 and, when
 *      keep_host is not NULL, keep_host [B, q_start_pos/cpu_block_tokens]
 *      (out, host; needs dev->keep).
 *
 * flags: BSX_FORCE_FIRST_LAST as for bsx_map_mask_to_cpu_blocks.
 * BSX_STEP_OFFLOAD attends as the pages' offload mode does (the keep flags,
 * then bsx_cpu_block_mask into dev->bsa_mask, and the split attention over
 * that mask); the pages' offload mode also sets BSX_FORCE_FIRST_LAST.
 * BSX_STEP_E4M3_ESTIMATE quantizes the uploaded q and k into dev->q8 and
 * dev->k8 (bsx_quantize_e4m3) and runs the estimate on them (bf16, d = 128).
 * BSX_STEP_FUSED replaces the split attention and the merge by one
 * bsx_bsa_prefill over every key block into (dev->o, dev->lse), as
 * bsx_chunk_prefill does (with q_start_pos = 0: whole-sequence prefill);
 * dev->o_curr and dev->lse_curr are then not used and may be NULL.  Without
 * BSX_STEP_OFFLOAD and BSX_STEP_E4M3_ESTIMATE the step then IS
 * bsx_chunk_prefill (one kernel where that call runs one, after all three
 * uploads), and dev->workspace must hold bsx_chunk_prefill_workspace_bytes().
 * With BSX_STEP_OFFLOAD and q_start_pos >= cpu_block_tokens, dev->keep is
 * required.
 *
 * Streams: the uploads go on `upload_stream` (q and k, then v), the launches
 * on `stream`, the read-back on `download_stream`; events order them (the
 * estimate waits for q and k, the attention for v as well, the read-back for
 * the launches), so v's upload overlaps the estimate, which does not read it.
 * upload_stream or download_stream NULL means `stream`.  When dev->done is
 * a CUDA event, the call first makes upload_stream and stream wait for it
 * and records it after the read-back: a caller that alternates two buffer
 * sets (each with its own event) on the same three streams overlaps one
 * step's uploads and read-back with the other step's launches, and no
 * buffer is written before the step that used it last has been read back.
 * The call returns without synchronising: the host outputs are valid once
 * download_stream has completed (or dev->done has), and the host buffers
 * must stay untouched until then.  Host buffers should be page-locked
 * (cudaHostAlloc / cudaHostRegister) for the copies to be asynchronous.
 *
 * Every argument is validated before anything is enqueued (as the entry
 * points above validate theirs); a CUDA error after that returns
 * BSX_ERR_CUDA and may leave part of the step enqueued.
 */
int bsx_chunk_step_host(bsx_shape s, const void* q_host, const void* k_host,
                        const void* v_host, int q_len, int q_start_pos, int stride,
                        float threshold, int cpu_block_tokens, int flags,
                        const bsx_chunk_buffers* dev, void* o_host, float* lse_host,
                        uint8_t* keep_host, void* stream, void* upload_stream,
                        void* download_stream);

/*
 * Test hook for the failure path (not for production use).  Arms, for the
 * calling host thread only, the next bf16 bsx_bsa_prefill or
 * bsx_bsa_prefill_split launch (including those made by bsx_chunk_step_host,
 * and by bsx_chunk_prefill when it does not run as one fused kernel): in CTA
 * `cta` of that launch (its linear grid
 * index; CTA 0 is the last 128-row query tile of head 0 of batch 0 in the
 * first key-block range) the copy producer stops before K/V ring item
 * `item` (items in the order the tensor pipe consumes them: K_0, K_1, V_0,
 * K_2, V_1, ...), with no copy and no arrival.  That CTA's waits for the item
 * then run out after their bound (about 2 s), the CTA drains its own copies
 * and MMAs, frees its tensor memory and exits without writing its O and
 * LSE, and the device error word records the attention kernel and the
 * wait that gave up (bsx_last_error).  Other CTAs are not affected.  The
 * launch consumes the setting; cta < 0 disarms it.  BSX_ERR_INVALID_ARG for
 * cta >= 0 with item < 0.
 */
int bsx_debug_drop_ring_item(int cta, int item);

/*
 * Test hook for the failure path of the fused chunk step (not for production
 * use).  Arms, for the calling host thread only, its next bsx_chunk_prefill
 * that runs as one kernel: selection row `row` (row = (b * Hq + h) * (q_len /
 * 128) + qb) writes its mask but never marks it ready, so that row's
 * attention CTA's bounded wait runs out (about 2 s); it then writes o = 0 and
 * lse = -inf for its rows, and the device error word records kernel id 3
 * (the fused step), wait site 1 (bsx_last_error).  The other rows are not
 * affected.  The call consumes the setting; row < 0 disarms it.  Returns
 * BSX_OK.
 */
int bsx_debug_fused_skip_row(int row);

/*
 * Asynchronous error status of the device.  Waits
 * for `stream` (a cudaStream_t; NULL is the legacy default stream, which also
 * waits for the blocking streams), then reads and clears the device error
 * word of the current device: the word in which a kernel records the first
 * bounded device wait that expired (the word is per device, so it reports
 * kernels of any stream that finished before the read; synchronise those
 * streams first to cover them).  Returns BSX_OK when the word was clear,
 * BSX_ERR_TIMEOUT when it was set, BSX_ERR_CUDA when a CUDA call failed
 * (the message goes to stderr).  Not for the hot path: it synchronises.
 */
int bsx_last_error(void* stream);

/*
 * The raw error word read by the calling host thread's last bsx_last_error
 * call (0 = none; otherwise bit 31 set, bits 0..7 the kernel: 1 = tcgen05
 * attention, 2 = tcgen05 estimator (both also inside the fused chunk step),
 * 3 = the fused chunk step's hand-over between its stages; bits 8..15 the
 * wait that gave up; for kernel 3: 1 = an attention CTA's wait for its
 * row's mask, 2 = a selection's wait for its estimate tiles, 3 = a worker's
 * tile-id ring).
 */
unsigned int bsx_last_error_code(void);

#ifdef __cplusplus
}
#endif

#endif /* BSXATTN_H_ */
