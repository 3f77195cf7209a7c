// C ABI of the library: argument validation, kernel choice, launches.
// Declarations and the meaning of every argument: include/bsxattn.h.
#include <limits.h>
#include <math.h>
#include <stdio.h>

#include <atomic>

#include "../../include/bsxattn.h"
#include "common.cuh"
#include "launchers.h"

namespace {

// Device error word (one per device that loads the library).  Kernels that
// run bounded waits record which wait gave up; bsx_last_error reads it.
__device__ unsigned g_bsx_err_word = 0;

constexpr int kMaxDevices = 64;
std::atomic<unsigned*> g_err_ptr[kMaxDevices];

// Device address of the error word for the current device (looked up once
// per device; host code cannot use the symbol itself as an address).  The
// cached address belongs to the device's primary context (the runtime API's
// context) and does not survive cudaDeviceReset.
unsigned* err_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  unsigned* w = g_err_ptr[dev].load(std::memory_order_acquire);
  if (!w) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bsx_err_word) != cudaSuccess) return nullptr;
    w = static_cast<unsigned*>(p);
    g_err_ptr[dev].store(w, std::memory_order_release);
  }
  return w;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Common shape checks; fills the internal problem description.
// e4m3 operands are accepted only where `allow_e4m3` (the estimate), with d = 128.
// Calls that work on the block mask (`masked`) also need its element count
// B * Hq * (q_len/128) * (Lk/128) to fit a 32-bit int: their grids and tile
// indices are 32-bit.
int make_problem(const bsx_shape& s, int q_len, int q_start_pos, bsx::Problem* p,
                 bool allow_e4m3 = false, bool masked = true) {
  if (s.B < 1 || s.Hq < 1 || s.Hkv < 1 || s.Hq % s.Hkv != 0) return BSX_ERR_INVALID_ARG;
  const bool e4m3 = s.dtype == BSX_F8E4M3 && allow_e4m3;
  if (s.dtype != BSX_F32 && s.dtype != BSX_BF16 && !e4m3) return BSX_ERR_UNSUPPORTED;
  if (s.d != 64 && s.d != 128) return BSX_ERR_UNSUPPORTED;
  if (e4m3 && s.d != 128) return BSX_ERR_UNSUPPORTED;
  if (q_len < 128 || q_len % 128 != 0) return BSX_ERR_INVALID_ARG;
  if (q_start_pos < 0 || q_start_pos % 128 != 0) return BSX_ERR_INVALID_ARG;
  const long long Lk = (long long)q_start_pos + q_len;
  if (Lk > (1LL << 24)) return BSX_ERR_UNSUPPORTED;
  p->B = s.B;
  p->Hq = s.Hq;
  p->Hkv = s.Hkv;
  p->d = s.d;
  p->dtype = s.dtype;
  p->q_len = q_len;
  p->q_start_pos = q_start_pos;
  p->Lk = (int)Lk;
  p->nqb = q_len / 128;
  p->nkb = (int)(Lk / 128);
  if (masked && (long long)s.B * s.Hq * p->nqb * p->nkb > INT_MAX) return BSX_ERR_UNSUPPORTED;
  return BSX_OK;
}

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return BSX_OK;
  fprintf(stderr, "bsxattn: CUDA error %s\n", cudaGetErrorString(e));
  return BSX_ERR_CUDA;
}

constexpr int kMaxKeyBlocks = 8192;  // selection sorts up to this many blocks per row

// Failure-path test hook (bsx_debug_drop_ring_item): armed per host thread,
// consumed by the next tcgen05 attention launch of that thread.
thread_local bsx::BsaDrop t_drop;

// The raw error word the calling thread's last bsx_last_error read.
thread_local unsigned t_last_word = 0;

// Failure-path test hook of the fused chunk step (bsx_debug_fused_skip_row):
// armed per host thread, consumed by its next fused step.
thread_local int t_skip_row = -1;

size_t round_up_256(size_t n) { return (n + 255) / 256 * 256; }

bsx::BsaDrop take_drop() {
  const bsx::BsaDrop d = t_drop;
  t_drop = bsx::BsaDrop();
  return d;
}

}  // namespace

extern "C" {

int bsx_version(void) { return (0 << 16) | 1; }

const char* bsx_status_string(int status) {
  switch (status) {
    case BSX_OK: return "ok";
    case BSX_ERR_INVALID_ARG: return "invalid argument";
    case BSX_ERR_UNSUPPORTED: return "unsupported dtype, head dim or stride";
    case BSX_ERR_CUDA: return "CUDA error";
    case BSX_ERR_TIMEOUT: return "a bounded device wait expired";
    case BSX_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
  }
}

size_t bsx_estimate_workspace_bytes(bsx_shape s, int q_len, int q_start_pos, int stride) {
  bsx::Problem p;
  if (make_problem(s, q_len, q_start_pos, &p, true) != BSX_OK) return 0;
  if (stride != 4 && stride != 8 && stride != 16) return 0;
  return (size_t)p.B * p.Hq * p.nkb * (size_t)(q_len / stride) * sizeof(float);
}

int bsx_xattn_estimate(bsx_shape s, const void* q, const void* k, int q_len,
                       int q_start_pos, int stride, float threshold, uint8_t* mask,
                       float* block_sums, void* workspace, size_t workspace_bytes,
                       void* stream) {
  bsx::Problem p;
  int rc = make_problem(s, q_len, q_start_pos, &p, true);
  if (rc != BSX_OK) return rc;
  if (stride != 4 && stride != 8 && stride != 16) return BSX_ERR_UNSUPPORTED;
  if (!(threshold > 0.0f) || isnan(threshold)) return BSX_ERR_INVALID_ARG;
  if (!q || !k || !mask || !aligned16(q) || !aligned16(k)) return BSX_ERR_INVALID_ARG;
  if (block_sums && !aligned16(block_sums)) return BSX_ERR_INVALID_ARG;
  if (p.nkb > kMaxKeyBlocks) return BSX_ERR_UNSUPPORTED;
  const size_t need = bsx_estimate_workspace_bytes(s, q_len, q_start_pos, stride);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return BSX_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float* lse_part = static_cast<float*>(workspace);
  cudaError_t e = p.dtype == BSX_F32
                      ? bsx::launch_estimate_simt(p, q, k, stride, lse_part, st)
                      : bsx::launch_estimate_tc(p, q, k, stride, lse_part, err_word(), st);
  if (e != cudaSuccess) return cuda_status(e);
  e = bsx::launch_select(p, stride, threshold, lse_part, mask, block_sums, st);
  return cuda_status(e);
}

int bsx_bsa_prefill(bsx_shape s, const void* q, const void* k, const void* v,
                    const uint8_t* mask, int q_len, int q_start_pos, int kb_begin,
                    int kb_end, void* o, float* lse, void* stream) {
  bsx::Problem p;
  int rc = make_problem(s, q_len, q_start_pos, &p);
  if (rc != BSX_OK) return rc;
  if (kb_begin < 0 || kb_begin > kb_end || kb_end > p.nkb) return BSX_ERR_INVALID_ARG;
  if (!q || !k || !v || !mask || !o || !lse) return BSX_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return BSX_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (p.dtype == BSX_BF16) {
    // tcgen05 path: one 128-row q-tile per CTA, up to kMaxKeyBlocks per row
    if (kb_end - kb_begin > kMaxKeyBlocks) return BSX_ERR_UNSUPPORTED;
    const bsx::BsaRange r{kb_begin, kb_end, o, lse};
    e = bsx::launch_bsa_tc(p, q, k, v, mask, 1, &r, err_word(), st, take_drop());
  } else {
    e = bsx::launch_bsa_simt(p, q, k, v, mask, kb_begin, kb_end, o, lse, st);
  }
  return cuda_status(e);
}

int bsx_bsa_prefill_split(bsx_shape s, const void* q, const void* k, const void* v,
                          const uint8_t* mask, int q_len, int q_start_pos, void* o_hist,
                          float* lse_hist, void* o_curr, float* lse_curr, void* stream) {
  bsx::Problem p;
  int rc = make_problem(s, q_len, q_start_pos, &p);
  if (rc != BSX_OK) return rc;
  if (!q || !k || !v || !mask || !o_hist || !lse_hist || !o_curr || !lse_curr)
    return BSX_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o_hist) ||
      !aligned16(lse_hist) || !aligned16(o_curr) || !aligned16(lse_curr))
    return BSX_ERR_INVALID_ARG;
  const int cur = q_start_pos / 128;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (p.dtype == BSX_BF16) {
    if (cur > kMaxKeyBlocks || p.nkb - cur > kMaxKeyBlocks) return BSX_ERR_UNSUPPORTED;
    // history CTAs (the long ones) first, the current chunk's fill the tail
    const bsx::BsaRange r[2] = {{0, cur, o_hist, lse_hist}, {cur, p.nkb, o_curr, lse_curr}};
    e = bsx::launch_bsa_tc(p, q, k, v, mask, 2, r, err_word(), st, take_drop());
  } else {
    e = bsx::launch_bsa_simt(p, q, k, v, mask, 0, cur, o_hist, lse_hist, st);
    if (e == cudaSuccess)
      e = bsx::launch_bsa_simt(p, q, k, v, mask, cur, p.nkb, o_curr, lse_curr, st);
  }
  return cuda_status(e);
}

int bsx_quantize_e4m3(const void* src, uint8_t* dst, long long n, void* stream) {
  if (n < 0 || (n > 0 && (!src || !dst))) return BSX_ERR_INVALID_ARG;
  return cuda_status(bsx::launch_quantize_e4m3(src, dst, n, static_cast<cudaStream_t>(stream)));
}

int bsx_merge_attn(bsx_shape s, int q_len, void* o1, float* lse1, const void* o2,
                   const float* lse2, void* stream) {
  bsx::Problem p;
  int rc = make_problem(s, q_len, 0, &p, false, false);
  if (rc != BSX_OK) return rc;
  if (!o1 || !lse1 || !o2 || !lse2) return BSX_ERR_INVALID_ARG;
  if (!aligned16(o1) || !aligned16(o2)) return BSX_ERR_INVALID_ARG;
  return cuda_status(bsx::launch_merge(p, o1, lse1, o2, lse2, static_cast<cudaStream_t>(stream)));
}

int bsx_map_mask_to_cpu_blocks(bsx_shape s, const uint8_t* mask, int q_len,
                               int q_start_pos, int cpu_block_tokens, int flags,
                               uint8_t* keep, void* stream) {
  bsx::Problem p;
  int rc = make_problem(s, q_len, q_start_pos, &p);
  if (rc != BSX_OK) return rc;
  if (cpu_block_tokens < 128 || cpu_block_tokens % 128 != 0) return BSX_ERR_INVALID_ARG;
  if (q_start_pos % cpu_block_tokens != 0) return BSX_ERR_INVALID_ARG;
  if ((flags & ~BSX_FORCE_FIRST_LAST) != 0) return BSX_ERR_INVALID_ARG;
  const int n_cpu = q_start_pos / cpu_block_tokens;
  if (n_cpu > 0 && (!mask || !keep)) return BSX_ERR_INVALID_ARG;
  return cuda_status(bsx::launch_map(p, mask, cpu_block_tokens, flags, keep,
                                     static_cast<cudaStream_t>(stream)));
}

size_t bsx_chunk_prefill_workspace_bytes(bsx_shape s, int q_len, int q_start_pos,
                                         int stride) {
  const size_t est = bsx_estimate_workspace_bytes(s, q_len, q_start_pos, stride);
  if (est == 0) return 0;
  bsx::Problem p;
  if (make_problem(s, q_len, q_start_pos, &p, true) != BSX_OK) return 0;
  return round_up_256(est) + bsx::fused_ctl_bytes(p, stride);
}

int bsx_chunk_prefill(bsx_shape s, const void* q, const void* k, const void* v, int q_len,
                      int q_start_pos, int stride, float threshold, uint8_t* mask, void* o,
                      float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  // validate everything before the first launch, so nothing is enqueued on error
  bsx::Problem p;
  int rc = make_problem(s, q_len, q_start_pos, &p);
  if (rc != BSX_OK) return rc;
  if (stride != 4 && stride != 8 && stride != 16) return BSX_ERR_UNSUPPORTED;
  if (!(threshold > 0.0f) || isnan(threshold)) return BSX_ERR_INVALID_ARG;
  if (!q || !k || !v || !mask || !o || !lse) return BSX_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return BSX_ERR_INVALID_ARG;
  if (p.nkb > kMaxKeyBlocks) return BSX_ERR_UNSUPPORTED;
  const size_t need = bsx_chunk_prefill_workspace_bytes(s, q_len, q_start_pos, stride);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return BSX_ERR_WORKSPACE;
  if (bsx::fused_step_supported(p, stride)) {
    // one kernel: estimate, selection and attention (the control block after
    // the partials)
    const size_t off = round_up_256(bsx_estimate_workspace_bytes(s, q_len, q_start_pos, stride));
    unsigned* ctl = reinterpret_cast<unsigned*>(static_cast<char*>(workspace) + off);
    const int skip = t_skip_row;
    t_skip_row = -1;
    const bsx::FusedOut out{mask, o, lse, nullptr, nullptr, nullptr, 0};
    return cuda_status(bsx::launch_fused_step(p, q, k, v, stride, threshold,
                                              static_cast<float*>(workspace), ctl, need - off,
                                              out, err_word(), skip,
                                              static_cast<cudaStream_t>(stream)));
  }
  rc = bsx_xattn_estimate(s, q, k, q_len, q_start_pos, stride, threshold, mask, nullptr,
                          workspace, workspace_bytes, stream);
  if (rc != BSX_OK) return rc;
  return bsx_bsa_prefill(s, q, k, v, mask, q_len, q_start_pos, 0, p.nkb, o, lse, stream);
}

int bsx_chunk_step(bsx_shape s, const void* q, const void* k, const void* v, int q_len,
                   int q_start_pos, int stride, float threshold, int cpu_block_tokens,
                   uint8_t* mask, void* o, float* lse, void* o_curr, float* lse_curr,
                   uint8_t* keep, void* workspace, size_t workspace_bytes, void* stream) {
  // validate everything before the first launch, so nothing is enqueued on error
  bsx::Problem p;
  int rc = make_problem(s, q_len, q_start_pos, &p);
  if (rc != BSX_OK) return rc;
  if (stride != 4 && stride != 8 && stride != 16) return BSX_ERR_UNSUPPORTED;
  if (!(threshold > 0.0f) || isnan(threshold)) return BSX_ERR_INVALID_ARG;
  if (!q || !k || !v || !mask || !o || !lse || !o_curr || !lse_curr) return BSX_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      !aligned16(o_curr) || !aligned16(lse_curr))
    return BSX_ERR_INVALID_ARG;
  const int cur = q_start_pos / 128;
  if (cur > kMaxKeyBlocks || p.nkb - cur > kMaxKeyBlocks) return BSX_ERR_UNSUPPORTED;
  const bool map = keep != nullptr && q_start_pos >= cpu_block_tokens;
  if (keep && (cpu_block_tokens < 128 || cpu_block_tokens % 128 != 0 ||
               q_start_pos % cpu_block_tokens != 0))
    return BSX_ERR_INVALID_ARG;
  const size_t need = bsx_chunk_prefill_workspace_bytes(s, q_len, q_start_pos, stride);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return BSX_ERR_WORKSPACE;
  if (bsx::fused_step_supported(p, stride)) {
    // one kernel: estimate, selection (and the CPU-block flags), attention on
    // the history and on the current chunk, merge
    const size_t off = round_up_256(bsx_estimate_workspace_bytes(s, q_len, q_start_pos, stride));
    unsigned* ctl = reinterpret_cast<unsigned*>(static_cast<char*>(workspace) + off);
    const int skip = t_skip_row;
    t_skip_row = -1;
    // with no history (q_start_pos 0) the step is the current chunk alone
    const bsx::FusedOut out{mask,
                            o,
                            lse,
                            q_start_pos > 0 ? o_curr : nullptr,
                            q_start_pos > 0 ? lse_curr : nullptr,
                            map ? keep : nullptr,
                            cpu_block_tokens};
    return cuda_status(bsx::launch_fused_step(p, q, k, v, stride, threshold,
                                              static_cast<float*>(workspace), ctl, need - off,
                                              out, err_word(), skip,
                                              static_cast<cudaStream_t>(stream)));
  }
  rc = bsx_xattn_estimate(s, q, k, q_len, q_start_pos, stride, threshold, mask, nullptr,
                          workspace, workspace_bytes, stream);
  if (rc == BSX_OK)
    rc = bsx_bsa_prefill_split(s, q, k, v, mask, q_len, q_start_pos, o, lse, o_curr, lse_curr,
                               stream);
  if (rc == BSX_OK) rc = bsx_merge_attn(s, q_len, o, lse, o_curr, lse_curr, stream);
  if (rc == BSX_OK && map)
    rc = bsx_map_mask_to_cpu_blocks(s, mask, q_len, q_start_pos, cpu_block_tokens, 0, keep,
                                    stream);
  return rc;
}

int bsx_cpu_block_mask(bsx_shape s, const uint8_t* keep, int q_len, int q_start_pos,
                       int cpu_block_tokens, uint8_t* mask, void* stream) {
  bsx::Problem p;
  int rc = make_problem(s, q_len, q_start_pos, &p);
  if (rc != BSX_OK) return rc;
  if (cpu_block_tokens < 128 || cpu_block_tokens % 128 != 0) return BSX_ERR_INVALID_ARG;
  if (q_start_pos % cpu_block_tokens != 0) return BSX_ERR_INVALID_ARG;
  if (!mask || (q_start_pos > 0 && !keep)) return BSX_ERR_INVALID_ARG;
  return cuda_status(bsx::launch_cpu_block_mask(p, keep, cpu_block_tokens, mask,
                                                static_cast<cudaStream_t>(stream)));
}

int bsx_debug_drop_ring_item(int cta, int item) {
  if (cta >= 0 && item < 0) return BSX_ERR_INVALID_ARG;
  t_drop.cta = cta < 0 ? -1 : cta;
  t_drop.item = cta < 0 ? -1 : item;
  return BSX_OK;
}

int bsx_debug_fused_skip_row(int row) {
  t_skip_row = row < 0 ? -1 : row;
  return BSX_OK;
}

int bsx_last_error(void* stream) {
  t_last_word = 0;
  unsigned* w = err_word();
  if (!w) return BSX_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_status(e);
  unsigned h = 0;
  e = cudaMemcpyAsync(&h, w, sizeof(h), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_status(e);
  if (h != 0) {
    e = cudaMemsetAsync(w, 0, sizeof(unsigned), st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_status(e);
  }
  t_last_word = h;
  return h ? BSX_ERR_TIMEOUT : BSX_OK;
}

unsigned int bsx_last_error_code(void) { return t_last_word; }

}  // extern "C"
