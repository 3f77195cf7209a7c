// bsx_chunk_step_host: one chunk step from host buffers to host buffers.
// Uploads, the step's launches and the read-back are all enqueued here, each
// on its own stream and ordered by events, so that a caller alternating two
// buffer sets overlaps one step's copies with the other step's launches.
#include <stdio.h>

#include "../../include/bsxattn.h"
#include "common.cuh"
#include "launchers.h"

namespace {

bool a16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// BSX_STEP_FUSED without the offload mask or e4m3 estimate operands runs as
// bsx_chunk_prefill, one kernel where the problem allows it.  (The split
// step keeps its separate launches: as one kernel, bsx_chunk_step, it
// measured the same.)
bool one_kernel(const bsx_shape& s, int q_len, int P, int stride, int flags) {
  if (!(flags & BSX_STEP_FUSED) || (flags & (BSX_STEP_OFFLOAD | BSX_STEP_E4M3_ESTIMATE)))
    return false;
  bsx::Problem p{};
  p.dtype = s.dtype;
  p.d = s.d;
  p.nkb = (P + q_len) / 128;
  return bsx::fused_step_supported(p, stride);
}

int cuda_fail(cudaError_t e) {
  fprintf(stderr, "bsxattn: CUDA error %s\n", cudaGetErrorString(e));
  return BSX_ERR_CUDA;
}

// Every check the step's entry points make, done before the first enqueue.
int validate(const bsx_shape& s, const void* qh, const void* kh, const void* vh, int q_len,
             int P, int stride, float threshold, int cpu_tokens, int flags,
             const bsx_chunk_buffers* dev, const void* oh, const float* lh,
             const uint8_t* keep_host) {
  if (!dev || !qh || !kh || !vh || !oh || !lh) return BSX_ERR_INVALID_ARG;
  if (flags & ~(BSX_FORCE_FIRST_LAST | BSX_STEP_OFFLOAD | BSX_STEP_E4M3_ESTIMATE |
                BSX_STEP_FUSED))
    return BSX_ERR_INVALID_ARG;
  const bool fused = flags & BSX_STEP_FUSED;
  if (s.B < 1 || s.Hq < 1 || s.Hkv < 1 || s.Hq % s.Hkv != 0) return BSX_ERR_INVALID_ARG;
  if (s.dtype != BSX_F32 && s.dtype != BSX_BF16) return BSX_ERR_UNSUPPORTED;
  if (s.d != 64 && s.d != 128) return BSX_ERR_UNSUPPORTED;
  if (stride != 4 && stride != 8 && stride != 16) return BSX_ERR_UNSUPPORTED;
  if (!(threshold > 0.0f)) return BSX_ERR_INVALID_ARG;
  if (q_len < 128 || q_len % 128 != 0 || P < 0 || P % 128 != 0) return BSX_ERR_INVALID_ARG;
  if ((long long)P + q_len > (1LL << 24)) return BSX_ERR_UNSUPPORTED;
  if ((P + q_len) / 128 > 8192) return BSX_ERR_UNSUPPORTED;
  if (cpu_tokens < 128 || cpu_tokens % 128 != 0 || P % cpu_tokens != 0)
    return BSX_ERR_INVALID_ARG;
  if (keep_host && P / cpu_tokens > 0 && !dev->keep) return BSX_ERR_INVALID_ARG;
  if (!a16(dev->q) || !a16(dev->k) || !a16(dev->v) || !a16(dev->o) || !a16(dev->lse) ||
      !dev->mask)
    return BSX_ERR_INVALID_ARG;
  if (!fused && (!a16(dev->o_curr) || !a16(dev->lse_curr))) return BSX_ERR_INVALID_ARG;
  if ((flags & BSX_STEP_OFFLOAD) && P / cpu_tokens > 0 && !dev->keep) return BSX_ERR_INVALID_ARG;
  if ((flags & BSX_STEP_OFFLOAD) && !dev->bsa_mask) return BSX_ERR_INVALID_ARG;
  if (flags & BSX_STEP_E4M3_ESTIMATE) {
    if (s.dtype != BSX_BF16 || s.d != 128) return BSX_ERR_UNSUPPORTED;
    if (!a16(dev->q8) || !a16(dev->k8)) return BSX_ERR_INVALID_ARG;
  }
  const size_t need =
      one_kernel(s, q_len, P, stride, flags)
          ? bsx_chunk_prefill_workspace_bytes(s, q_len, P, stride)
          : bsx_estimate_workspace_bytes(
                bsx_shape{s.B, s.Hq, s.Hkv, s.d,
                          (flags & BSX_STEP_E4M3_ESTIMATE) ? BSX_F8E4M3 : s.dtype},
                q_len, P, stride);
  if (need == 0 || !a16(dev->workspace) || dev->workspace_bytes < need) return BSX_ERR_WORKSPACE;
  return BSX_OK;
}

}  // namespace

namespace {

// Events of one call, created with timing off and destroyed before the call
// returns: an event destroyed while its record is still pending is released
// once the device has passed it.
struct CallEvents {
  cudaEvent_t ev[3] = {nullptr, nullptr, nullptr};
  cudaError_t make(int n) {
    for (int i = 0; i < n; ++i) {
      cudaError_t e = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
  ~CallEvents() {
    for (cudaEvent_t e : ev)
      if (e) cudaEventDestroy(e);
  }
};

// `dst` waits for everything enqueued on `src` so far
cudaError_t follow(cudaStream_t dst, cudaStream_t src, cudaEvent_t ev) {
  cudaError_t e = cudaEventRecord(ev, src);
  return e == cudaSuccess ? cudaStreamWaitEvent(dst, ev, 0) : e;
}

// Read-back of O, LSE (and the keep flags) on `dn`, after the step's launches
// on `st`; then `done` is recorded on `dn`.
int read_back(const bsx_shape& s, const bsx_chunk_buffers* dev, int n_cpu, bool map,
              size_t o_bytes, size_t lse_bytes, void* o_host, float* lse_host,
              uint8_t* keep_host, cudaStream_t st, cudaStream_t dn, cudaEvent_t done,
              cudaEvent_t ev) {
  cudaError_t e = dn != st ? follow(dn, st, ev) : cudaSuccess;
  if (e == cudaSuccess) e = cudaMemcpyAsync(o_host, dev->o, o_bytes, cudaMemcpyDeviceToHost, dn);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(lse_host, dev->lse, lse_bytes, cudaMemcpyDeviceToHost, dn);
  if (e == cudaSuccess && keep_host && map)
    e = cudaMemcpyAsync(keep_host, dev->keep, (size_t)s.B * n_cpu, cudaMemcpyDeviceToHost, dn);
  if (e == cudaSuccess && done) e = cudaEventRecord(done, dn);
  return e == cudaSuccess ? BSX_OK : cuda_fail(e);
}

}  // namespace

extern "C" int bsx_chunk_step_host(bsx_shape s, const void* q_host, const void* k_host,
                                   const void* v_host, int q_len, int q_start_pos, int stride,
                                   float threshold, int cpu_block_tokens, int flags,
                                   const bsx_chunk_buffers* dev, void* o_host, float* lse_host,
                                   uint8_t* keep_host, void* stream, void* upload_stream,
                                   void* download_stream) {
  const int P = q_start_pos;
  int rc = validate(s, q_host, k_host, v_host, q_len, P, stride, threshold, cpu_block_tokens,
                    flags, dev, o_host, lse_host, keep_host);
  if (rc != BSX_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaStream_t up = upload_stream ? static_cast<cudaStream_t>(upload_stream) : st;
  cudaStream_t dn = download_stream ? static_cast<cudaStream_t>(download_stream) : st;
  cudaEvent_t done = static_cast<cudaEvent_t>(dev->done);
  const size_t elt = s.dtype == BSX_BF16 ? 2 : 4;
  const long long Lk = (long long)P + q_len;
  const size_t q_elems = (size_t)s.B * q_len * s.Hq * s.d;
  const size_t kv_elems = (size_t)s.B * Lk * s.Hkv * s.d;
  const size_t lse_bytes = (size_t)s.B * s.Hq * q_len * sizeof(float);
  const int n_cpu = P / cpu_block_tokens;
  const bool fused = flags & BSX_STEP_FUSED;
  const bool map = n_cpu > 0 && dev->keep != nullptr;
  CallEvents ev;  // [0] Q and K uploaded, [1] V uploaded, [2] results ready
  cudaError_t e = ev.make(3);
  if (e != cudaSuccess) return cuda_fail(e);

  // The previous step on these buffers has been read back before they are
  // written again (its compute read q, k, v; its read-back reads o, lse, keep).
  if (done) {
    e = cudaStreamWaitEvent(up, done, 0);
    if (e == cudaSuccess && st != up) e = cudaStreamWaitEvent(st, done, 0);
    if (e != cudaSuccess) return cuda_fail(e);
  }

  // uploads: Q and K first (the estimate needs them), V behind them, so that
  // V's copy overlaps the estimate, which does not read it
  e = cudaMemcpyAsync(dev->q, q_host, q_elems * elt, cudaMemcpyHostToDevice, up);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(dev->k, k_host, kv_elems * elt, cudaMemcpyHostToDevice, up);
  if (e == cudaSuccess && up != st) e = follow(st, up, ev.ev[0]);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(dev->v, v_host, kv_elems * elt, cudaMemcpyHostToDevice, up);
  if (e == cudaSuccess && up != st) e = cudaEventRecord(ev.ev[1], up);
  if (e != cudaSuccess) return cuda_fail(e);

  if (one_kernel(s, q_len, P, stride, flags)) {
    // the step in one launch, which reads V as well
    if (up != st && cudaStreamWaitEvent(st, ev.ev[1], 0) != cudaSuccess) return BSX_ERR_CUDA;
    rc = bsx_chunk_prefill(s, dev->q, dev->k, dev->v, q_len, P, stride, threshold, dev->mask,
                           dev->o, dev->lse, dev->workspace, dev->workspace_bytes, st);
    if (rc == BSX_OK && map)
      rc = bsx_map_mask_to_cpu_blocks(s, dev->mask, q_len, P, cpu_block_tokens,
                                      flags & BSX_FORCE_FIRST_LAST, dev->keep, st);
    if (rc != BSX_OK) return rc;
    return read_back(s, dev, n_cpu, map, q_elems * elt, lse_bytes, o_host, lse_host,
                     keep_host, st, dn, done, ev.ev[2]);
  }

  // estimate (on e4m3 copies of the uploaded Q and K when asked)
  const void* qe = dev->q;
  const void* ke = dev->k;
  bsx_shape se = s;
  if (flags & BSX_STEP_E4M3_ESTIMATE) {
    rc = bsx_quantize_e4m3(dev->q, dev->q8, (long long)q_elems, st);
    if (rc == BSX_OK) rc = bsx_quantize_e4m3(dev->k, dev->k8, (long long)kv_elems, st);
    qe = dev->q8;
    ke = dev->k8;
    se.dtype = BSX_F8E4M3;
  }
  if (rc == BSX_OK)
    rc = bsx_xattn_estimate(se, qe, ke, q_len, P, stride, threshold, dev->mask, nullptr,
                            dev->workspace, dev->workspace_bytes, st);
  if (rc == BSX_OK && up != st && cudaStreamWaitEvent(st, ev.ev[1], 0) != cudaSuccess)
    rc = BSX_ERR_CUDA;
  if (rc != BSX_OK) return rc;

  // attention: history and current chunk in one launch, then the LSE merge
  // (or, fused, every key block in one range: the same result by the merge
  // identity, without the merge)
  const int map_flags = flags & BSX_FORCE_FIRST_LAST;
  const uint8_t* attn_mask = dev->mask;
  if (flags & BSX_STEP_OFFLOAD) {
    if (map)
      rc = bsx_map_mask_to_cpu_blocks(s, dev->mask, q_len, P, cpu_block_tokens, map_flags,
                                      dev->keep, st);
    if (rc == BSX_OK)
      rc = bsx_cpu_block_mask(s, n_cpu > 0 ? dev->keep : nullptr, q_len, P, cpu_block_tokens,
                              dev->bsa_mask, st);
    attn_mask = dev->bsa_mask;
  }
  if (rc == BSX_OK && fused)
    rc = bsx_bsa_prefill(s, dev->q, dev->k, dev->v, attn_mask, q_len, P, 0, (int)(Lk / 128),
                         dev->o, dev->lse, st);
  if (rc == BSX_OK && !fused)
    rc = bsx_bsa_prefill_split(s, dev->q, dev->k, dev->v, attn_mask, q_len, P, dev->o, dev->lse,
                               dev->o_curr, dev->lse_curr, st);
  if (rc == BSX_OK && !fused)
    rc = bsx_merge_attn(s, q_len, dev->o, dev->lse, dev->o_curr, dev->lse_curr, st);
  if (rc == BSX_OK && !(flags & BSX_STEP_OFFLOAD) && map)
    rc = bsx_map_mask_to_cpu_blocks(s, dev->mask, q_len, P, cpu_block_tokens, map_flags,
                                    dev->keep, st);
  if (rc != BSX_OK) return rc;

  return read_back(s, dev, n_cpu, map, q_elems * elt, lse_bytes, o_host, lse_host,
                   keep_host, st, dn, done, ev.ev[2]);
}
